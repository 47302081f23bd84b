// Decode-shaped partial attention on the 5th-generation tensor cores of
// sm_103a (tcgen05 + TMEM + TMA), bf16 inputs, head_dim 128: a few query
// tokens of every query head of one kv head, packed into one 128-row tile,
// against one piece of a CP rank's K/V chunk.
//
// What one work item computes: the Pass-Q step of context-parallel attention
// for decode-shaped queries ("Scaling LLM Inference ...", techreport rewrite,
// section "Context Parallelism for Million-Token Contexts", Pass-Q bullet:
// the queries visit the ranks that hold K/V), as an fp32 partial (O, LSE)
// that the N-way merge combines afterwards:
//   s_ij = scale * q_i . k_j  for the piece's keys with kv_pos(j) <= q_pos(i),
//   LSE_i = log sum_j exp(s_ij),  O_i = sum_j exp(s_ij - LSE_i) v_j.
//
// Design (one CTA per SM, looping over work items):
//   tile row r = (token r / G, head hk * G + r % G) for the G = Hq / Hkv query
//   heads that read kv head hk (the Q tensor map's box is 64 x G x 128 / G);
//   warps 0..3   softmax: one thread per row (TMEM lane), exp2-domain online
//                softmax with a lazy rescale
//   warp 4       TMA producer: Q once per item, K_j / V_j into a 3-stage ring
//   warp 5       MMA issuer (one thread): S(j) = Q K_j^T into score buffer
//                j % 2, O += P(j) V_j with P from TMEM
// TMEM: score buffers at columns 0 and 128, O at 256, P buffers (bf16 pairs)
// at 384 and 448.  S(j + 2) is issued only after P(j) is ready (the softmax
// has read score buffer j % 2), and the softmax writes P buffer j % 2 for
// step j + 2 only after S(j + 2) is complete, whose commit covers the PV MMA
// of step j that read that buffer: no MMA ordering between different
// accumulators is assumed.
//
// Every mbarrier wait is bounded (AttnParams::wait_ns of global time); a wait
// that gives up records CPATTN_ERR_TIMEOUT in a device status word, the CTA
// drains its own copies and MMAs, frees its TMEM and returns without writing
// output.
#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>

#include <mutex>

#include "cpattn_internal.h"
#include "epilogue.cuh"
#include "tc_ptx.cuh"
#include "tmem_ldst.cuh"

namespace cpattn {

__device__ unsigned int g_attn_tc_status;

namespace {

using namespace tc;

constexpr int kBM = 128;                  // query rows per tile (TMEM lanes)
constexpr int kBN = 128;                  // keys per tile
constexpr int kD = 128;                   // head dim
constexpr int kBoxBytes = 128 * 128;      // 128 rows x 64 bf16 (one swizzle span)
constexpr int kTileBytes = 2 * kBoxBytes; // 128 x 128 bf16
constexpr int kStages = 3;
constexpr float kRescaleLog2 = 8.0f;      // lazy-rescale threshold (log2 units)
constexpr unsigned long long kDrainNs = 20000000ull;

struct Layout {
  static constexpr int kThreads = 6 * 32;
  static constexpr int kTmaWarp = 4;
  static constexpr int kMmaWarp = 5;
  static constexpr int kTmemCols = 512;
  static constexpr int t_s = 0, t_o = 256, t_p = 384;
  static constexpr int q_off = 0;
  static constexpr int k_off = q_off + kTileBytes;
  static constexpr int v_off = k_off + kStages * kTileBytes;
  static constexpr int bar_off = v_off + kStages * kTileBytes;
  static constexpr int b_qfull = 0;
  static constexpr int b_qempty = 1;  // the item's last QK MMA is done with Q
  static constexpr int b_kfull = 2;
  static constexpr int b_kempty = b_kfull + kStages;
  static constexpr int b_vfull = b_kempty + kStages;
  static constexpr int b_vempty = b_vfull + kStages;
  static constexpr int b_sfull = b_vempty + kStages;  // per score buffer
  static constexpr int b_pready = b_sfull + 2;        // per P buffer
  static constexpr int b_pvstep = b_pready + 2;       // every PV but an item's last
  static constexpr int b_ofull = b_pvstep + 1;        // an item's last PV
  static constexpr int b_ofree = b_ofull + 1;         // softmax warps have read O
  static constexpr int b_drain = b_ofree + 1;
  static constexpr int n_bars = b_drain + 1;
  static constexpr int tmem_slot_off = bar_off + n_bars * 8;
  static constexpr int abort_off = tmem_slot_off + 4;
  static constexpr int bytes = abort_off + 4;
  static constexpr int alloc_bytes = bytes + 1024;  // room to align the base to 1024
};

constexpr uint32_t kIdescQK = make_idesc(kBM, kBN, false);
constexpr uint32_t kIdescPV = make_idesc(kBM, kD, true);

static_assert(sizeof(AttnParams) + 3 * sizeof(CUtensorMap) <= 4096, "kernel parameters too large");

__global__ void __launch_bounds__(Layout::kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ AttnParams p) {
  using L = Layout;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int idx) -> uint32_t { return sb + L::bar_off + 8 * idx; };
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::abort_off);
  const unsigned long long wait_ns = p.wait_ns;
  auto wait = [&](uint32_t b, uint32_t parity) -> bool {
    return wait_phase<false>(b, parity, abort_flag, &g_attn_tc_status, wait_ns, true);
  };
  auto drain_wait = [&](uint32_t b, uint32_t parity) -> bool {
    return wait_phase<false>(b, parity, abort_flag, &g_attn_tc_status, kDrainNs, false);
  };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const PairDesc *pairs = p.pairs;
  const int n_pairs = p.n_pairs;
  const int G = p.pack_g;  // query heads per tile
  const int stride = (int)gridDim.x;

  // ---- setup (once per CTA)
  if (threadIdx.x == 0) {
    mbar_init(bar(L::b_qfull), 1);
    mbar_init(bar(L::b_qempty), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(L::b_kfull + s), 1);
      mbar_init(bar(L::b_kempty + s), 1);
      mbar_init(bar(L::b_vfull + s), 1);
      mbar_init(bar(L::b_vempty + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(L::b_sfull + b), 1);
      mbar_init(bar(L::b_pready + b), 4);
    }
    mbar_init(bar(L::b_pvstep), 1);
    mbar_init(bar(L::b_ofull), 1);
    mbar_init(bar(L::b_ofree), 4);
    mbar_init(bar(L::b_drain), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == L::kTmaWarp && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == L::kMmaWarp) {
    tmem_alloc_1(sb + L::tmem_slot_off, L::kTmemCols);
    tmem_relinquish_1();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + L::tmem_slot_off);

  // ---- work item geometry: (pair, kv split, kv head, batch)
  struct Item {
    const PairDesc *pd;
    int h0, hk, split, b, n_kv, n_unmasked;
    int64_t ks, ke;  // this item's keys [ks, ke) of the pair
  };
  auto decode = [&](int item, Item &it) {
    int lo = 0, hi = n_pairs - 1;  // last pair whose cta_begin <= item
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pairs[mid].cta_begin <= item) lo = mid; else hi = mid - 1;
    }
    const PairDesc &pd = pairs[lo];
    it.pd = &pd;
    int local = item - pd.cta_begin;
    it.hk = local % p.Hkv;
    local /= p.Hkv;
    it.split = local / p.B;
    it.b = local % p.B;
    it.h0 = it.hk * G;
    it.ks = (int64_t)it.split * p.kv_split;
    it.ke = it.ks + p.kv_split < pd.kv_len ? it.ks + p.kv_split : pd.kv_len;
    // Keys [ks, kv_end) are visible to some row of the tile; [ks, full_end) to every row.
    int64_t kv_end = it.ke, full_end = it.ke;
    if (p.causal) {
      const int64_t last_lim = (int64_t)(pd.q_len - 1) + pd.delta + 1;
      const int64_t first_lim = pd.delta + 1;
      kv_end = last_lim < kv_end ? last_lim : kv_end;
      full_end = first_lim < full_end ? first_lim : full_end;
    }
    if (kv_end < it.ks) kv_end = it.ks;
    if (full_end < it.ks) full_end = it.ks;
    it.n_kv = (int)((kv_end - it.ks + kBN - 1) / kBN);
    it.n_unmasked = (int)((full_end - it.ks) / kBN);
  };

  if (warp == L::kTmaWarp) {
    // ================================================= TMA producer
    // Loads in the order the MMA thread consumes them (Q, K_0, K_1, V_0, K_2,
    // V_1, ..., V_{n-1}); K/V steps count up across items.
    if (lane == 0) {
      int nk[kStages] = {0}, nv[kStages] = {0}, nq = 0;
      int g = 0, nitem = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < p.total_ctas && ok; item += stride) {
        Item it;
        decode(item, it);
        if (it.n_kv == 0) continue;
        if (nitem > 0 && !wait(bar(L::b_qempty), (nitem - 1) & 1)) { ok = false; break; }
        mbar_expect_tx(bar(L::b_qfull), kTileBytes);
        for (int half = 0; half < 2; ++half)
          tma_load_4d(sb + L::q_off + half * kBoxBytes, &tm_q, bar(L::b_qfull), half * 64, it.h0,
                      it.pd->q_row0, it.b);  // packed map: heads h0 .., rows q_row0 ..
        ++nq;
        auto load = [&](int full, int empty, int off, const CUtensorMap *map, int j,
                        int *count) -> bool {
          const int gj = g + j, st = gj % kStages;
          if (gj >= kStages && !wait(bar(empty + st), ((gj / kStages) - 1) & 1)) return false;
          mbar_expect_tx(bar(full + st), kTileBytes);
          const int row = it.pd->kv_row0 + (int)it.ks + j * kBN;
          for (int half = 0; half < 2; ++half)
            tma_load_4d(sb + off + st * kTileBytes + half * kBoxBytes, map, bar(full + st),
                        half * 64, it.hk, row, it.b);
          ++count[st];
          return true;
        };
        auto load_k = [&](int j) { return load(L::b_kfull, L::b_kempty, L::k_off, &tm_k, j, nk); };
        auto load_v = [&](int j) { return load(L::b_vfull, L::b_vempty, L::v_off, &tm_v, j, nv); };
        for (int j = 0; j < it.n_kv && ok; ++j) ok = load_k(j) && (j == 0 || load_v(j - 1));
        if (ok) ok = load_v(it.n_kv - 1);
        g += it.n_kv;
        ++nitem;
      }
      // Every copy this warp issued has landed before the CTA can exit (on
      // the normal path the MMA thread has consumed them all already; on an
      // abort the wait is short).
      {
        if (nq > 0) drain_wait(bar(L::b_qfull), (nq - 1) & 1);
        for (int s = 0; s < kStages; ++s) {
          if (nk[s] > 0) drain_wait(bar(L::b_kfull + s), (nk[s] - 1) & 1);
          if (nv[s] > 0) drain_wait(bar(L::b_vfull + s), (nv[s] - 1) & 1);
        }
      }
    }
    __syncwarp();
  } else if (warp == L::kMmaWarp) {
    // ================================================= MMA issuer (one thread)
    // Per item: S(0), S(1), then for every step j: O += P(j) V_j, S(j + 2).
    if (lane == 0) {
      const uint64_t dq0 = make_sdesc(sb + L::q_off, 16, 1024);
      const uint64_t dk0 = make_sdesc(sb + L::k_off, 16, 1024);
      const uint64_t dv0 = make_sdesc(sb + L::v_off, kBoxBytes, 1024);
      bool ok = true;
      int g = 0, nitem = 0;
      for (int item = blockIdx.x; item < p.total_ctas && ok; item += stride) {
        Item it;
        decode(item, it);
        const int n_kv = it.n_kv;
        if (n_kv == 0) continue;
        auto issue_qk = [&](int j) -> bool {
          const int gk = g + j, st = gk % kStages;
          if (!wait(bar(L::b_kfull + st), (gk / kStages) & 1)) return false;
          tc_fence_after();
          const uint64_t dk = dk0 + (uint64_t)((st * kTileBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) {
            const uint64_t off = (uint64_t)(((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4);
            mma_ss_1(tmem + L::t_s + (gk & 1) * 128, dq0 + off, dk + off, kIdescQK, kk > 0 ? 1u : 0u);
          }
          mma_commit_1(bar(L::b_sfull + (gk & 1)));
          mma_commit_1(bar(L::b_kempty + st));
          if (j == n_kv - 1) mma_commit_1(bar(L::b_qempty));  // the item's last QK
          return true;
        };
        if (!wait(bar(L::b_qfull), nitem & 1)) { ok = false; break; }
        ok = issue_qk(0) && (n_kv < 2 || issue_qk(1));
        for (int j = 0; j < n_kv && ok; ++j) {
          const int gj = g + j, sv = gj % kStages;
          if (!wait(bar(L::b_vfull + sv), (gj / kStages) & 1) ||
              !wait(bar(L::b_pready + (gj & 1)), (gj >> 1) & 1) ||
              (j == 0 && nitem > 0 && !wait(bar(L::b_ofree), (nitem - 1) & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t dv = dv0 + (uint64_t)((sv * kTileBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            mma_ts_1(tmem + L::t_o, tmem + L::t_p + (gj & 1) * 64 + kk * 8,
                     dv + (uint64_t)((kk * 16 * 128) >> 4), kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
          mma_commit_1(bar(L::b_vempty + sv));
          mma_commit_1(bar(j + 1 < n_kv ? L::b_pvstep : L::b_ofull));
          if (j + 2 < n_kv) ok = issue_qk(j + 2);
        }
        g += n_kv;
        ++nitem;
      }
      if (!ok) {
        mma_commit_1(bar(L::b_drain));
        drain_wait(bar(L::b_drain), 0);
      }
    }
    __syncwarp();
  } else {
    // ================================================= softmax warps
    const int r = warp * 32 + lane;  // row in the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const uint32_t t_s = tmem + lane_off + L::t_s;  // + 128 * buffer
    const uint32_t t_o = tmem + lane_off + L::t_o;
    const uint32_t t_p = tmem + lane_off + L::t_p;  // + 64 * buffer
    const float sl2 = p.scale_log2;
    bool ok = true;
    int g = 0, nitem = 0, pv_phase = 0;
    for (int item = blockIdx.x; item < p.total_ctas && ok; item += stride) {
      Item it;
      decode(item, it);
      const PairDesc &pd = *it.pd;
      const int n_kv = it.n_kv;
      const int qrow = r / G;             // token of this tile row
      const int head = it.h0 + r % G;
      const bool valid = qrow < pd.q_len;
      int64_t lim = it.ke;  // this row's visible keys: [ks, lim)
      if (p.causal) {
        const int64_t c = (int64_t)qrow + pd.delta + 1;
        lim = c < lim ? c : lim;
      }
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = 0; j < n_kv; ++j) {
        const int gj = g + j, buf = gj & 1;
        // Warp-uniform outcome: the TMEM accesses below are warp-collective.
        if (!__all_sync(0xffffffffu, wait(bar(L::b_sfull + buf), (gj >> 1) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[128];
        tmem_ld_x128(t_s + buf * 128, sr);
        float s[128];
#pragma unroll
        for (int c = 0; c < kBN; ++c) s[c] = __uint_as_float(sr[c]);
        if (j >= it.n_unmasked) {
          const int64_t nv = lim - it.ks - (int64_t)j * kBN;
          const int nvis = nv < 0 ? 0 : (nv > kBN ? kBN : (int)nv);
#pragma unroll
          for (int c = 0; c < kBN; ++c)
            if (c >= nvis) s[c] = -INFINITY;
        }
        float mk[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          float m = fmax3(s[k], s[k + 8], s[k + 16]);
#pragma unroll
          for (int i = 3; i < 15; i += 2) m = fmax3(m, s[k + 8 * i], s[k + 8 * (i + 1)]);
          mk[k] = fmaxf(m, s[k + 120]);
        }
        const float mx = fmax3(fmax3(mk[0], mk[1], mk[2]), fmax3(mk[3], mk[4], mk[5]),
                               fmaxf(mk[6], mk[7]));
        const float m_new = fmaxf(m_run, mx * sl2);
        const bool grow = m_new > m_run + kRescaleLog2;
        float alpha = 1.f;
        if (grow) {
          alpha = ex2(m_run - m_new);  // 0 when m_run = -inf
          l_run *= alpha;
        }
        const bool rescale_o = grow && (m_run != -INFINITY) && j > 0;
        if (grow) m_run = m_new;
        if (__any_sync(0xffffffffu, rescale_o)) {
          // O holds the PV of step j - 1 only once that MMA is complete.
          if (!__all_sync(0xffffffffu, wait(bar(L::b_pvstep), (pv_phase + j - 1) & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float a = rescale_o ? alpha : 1.f;
#pragma unroll 1
          for (int cc = 0; cc < kD / 8; ++cc) {
            uint32_t ov[8];
            tmem_ld_x8(t_o + cc * 8, ov);
#pragma unroll
            for (int x = 0; x < 8; ++x) ov[x] = __float_as_uint(__uint_as_float(ov[x]) * a);
            tmem_st_x8(t_o + cc * 8, ov);
          }
        }
        const float neg_m = m_run == -INFINITY ? 0.f : -m_run;
        const float2 sl2v = make_float2(sl2, sl2);
        const float2 negm = make_float2(neg_m, neg_m);
        float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                         make_float2(0.f, 0.f)};
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          uint32_t pk[16];
#pragma unroll
          for (int c = qq * 32; c < qq * 32 + 32; c += 2) {
            const float2 x = __ffma2_rn(make_float2(s[c], s[c + 1]), sl2v, negm);
            const float2 pv = make_float2(ex2(x.x), ex2(x.y));
            acc[(c >> 1) & 3] = __fadd2_rn(acc[(c >> 1) & 3], pv);
            pk[(c >> 1) - qq * 16] = pack_bf16(pv.x, pv.y);
          }
          tmem_st_x16(t_p + buf * 64 + qq * 16, pk);
        }
        const float2 a01 = __fadd2_rn(acc[0], acc[1]);
        const float2 a23 = __fadd2_rn(acc[2], acc[3]);
        const float2 a03 = __fadd2_rn(a01, a23);
        l_run += a03.x + a03.y;
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::b_pready + buf));
      }
      if (!ok) break;

      // ---- epilogue: O / l and LSE into the item's fp32 partial slot
      if (n_kv > 0) {
        if (!__all_sync(0xffffffffu, wait(bar(L::b_ofull), nitem & 1))) { ok = false; break; }
        tc_fence_after();
      }
      const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
      const float lse = l_run > 0.f ? (m_run + log2f(l_run)) * 0.6931471805599453f : -INFINITY;
      RowSink sink;
      if (valid) sink.init(p, pd, it.b, head, qrow, lse, true, pd.slot + it.split, nullptr, &g_attn_tc_status);
#pragma unroll 1
      for (int cc = 0; cc < kD / 32; ++cc) {
        float ov[32];
        if (n_kv > 0) {
          uint32_t raw[32];
          tmem_ld_x32(t_o + cc * 32, raw);
#pragma unroll
          for (int x = 0; x < 32; ++x) ov[x] = __uint_as_float(raw[x]) * inv_l;
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x) ov[x] = 0.f;
        }
        if (valid) sink.put<32>(cc * 32, ov);
      }
      if (n_kv > 0) {
        // O has been read: the next item's first PV may overwrite it.
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::b_ofree));
        pv_phase += n_kv - 1;
        ++nitem;
      }
      g += n_kv;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == L::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc_1(tmem, L::kTmemCols);
  }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(ptr);
    return nullptr;
  }();
  return fn;
}

// [b, s, h, d] bf16 view -> 4-D tensor map (d, h, s, b), box 64 x box_h x box_s x 1
// (box_h * box_s = 128 rows of 128 bytes each).
bool make_map(CUtensorMap *map, const void *base, int64_t B, int64_t S, int64_t H, int64_t D,
              int64_t sb, int64_t ss, int64_t sh, uint32_t box_h, uint32_t box_s) {
  EncodeTiledFn enc = get_encode_fn();
  if (enc == nullptr) return false;
  if (B == 1) sb = S * ss > 0 ? S * ss : 8;  // unused extent: any legal stride
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)S, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)sh * 2, (cuuint64_t)ss * 2, (cuuint64_t)sb * 2};
  cuuint32_t box[4] = {64, box_h, box_s, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

bool attn_decode_tc_supported(const AttnParams &p) {
  // The group fills whole TMA boxes, every query row of a pair fits in one
  // 128-row tile, and splits are whole KV tiles.
  if (p.in_f32 || p.D != kD || p.q_rows_total <= 0 || p.kv_rows_total <= 0) return false;
  if (p.pack_g <= 0 || p.pack_g != p.Hq / p.Hkv || kBM % p.pack_g != 0 || p.kv_split <= 0 ||
      p.kv_split % kBN)
    return false;
  for (int x = 0; x < p.n_pairs; ++x)
    if (p.pairs[x].q_len > kBM / p.pack_g) return false;
  return true;
}

cudaError_t launch_attn_decode_tc(AttnParams &p, cudaStream_t stream) {
  using L = Layout;
  int total = 0;
  for (int x = 0; x < p.n_pairs; ++x) {  // n_qtiles counts kv splits here
    PairDesc &pd = p.pairs[x];
    pd.n_qtiles = (pd.kv_len + p.kv_split - 1) / p.kv_split;
    pd.cta_begin = total;
    total += pd.n_qtiles * p.Hkv * p.B;
  }
  p.total_ctas = total;
  if (total == 0) return cudaSuccess;
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, p.q, p.B, p.q_rows_total, p.Hq, kD, p.q_sb, p.q_ss, p.q_sh,
                (uint32_t)p.pack_g, (uint32_t)(kBM / p.pack_g)) ||
      !make_map(&mk, p.k, p.B, p.kv_rows_total, p.Hkv, kD, p.k_sb, p.k_ss, p.k_sh, 1, kBN) ||
      !make_map(&mv, p.v, p.B, p.kv_rows_total, p.Hkv, kD, p.v_sb, p.v_ss, p.v_sh, 1, kBN))
    return cudaErrorInvalidValue;
  // Per device, once: the shared-memory attribute and the SM count.
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static bool configured[kMaxDevices] = {};
  static int sms[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return cudaErrorInvalidDevice;
  int sm_count = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!configured[dev]) {
      cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           L::alloc_bytes);
      if (e != cudaSuccess) return e;
      e = cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return e;
      configured[dev] = true;
    }
    sm_count = sms[dev];
  }
  // One CTA per SM (shared memory admits only one), each looping over items.
  const int grid = sm_count < total ? sm_count : total;
  p.persistent_ctas = grid;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(L::kThreads);
  cfg.dynamicSmemBytes = L::alloc_bytes;
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, attn_tc_kernel, mq, mk, mv, p);
}

unsigned int attn_tc_read_status(bool clear, cudaError_t *err) {
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_attn_tc_status, sizeof(v));
  if (e == cudaSuccess && clear) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_attn_tc_status, &zero, sizeof(zero));
  }
  if (err) *err = e;
  return v;
}

}  // namespace cpattn
