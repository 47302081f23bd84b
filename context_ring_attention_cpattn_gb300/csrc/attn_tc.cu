// Partial attention of (Q-chunk, KV-chunk) pairs on the 5th-generation tensor
// cores of sm_103a (tcgen05 + TMEM + TMA), bf16 inputs, head_dim 128.
//
// What one pair computes: the per-rank step of context-parallel ring
// attention ("Scaling LLM Inference ...", techreport rewrite, section
// "Context Parallelism for Million-Token Contexts", Pass-KV / Pass-Q bullets;
// the pages name only "a fast attention kernel" and give no design):
//   s_ij = scale * q_i . k_j  for keys with kv_pos(j) <= q_pos(i) (causal),
//   LSE_i = log sum_j exp(s_ij),  O_i = sum_j exp(s_ij - LSE_i) v_j,
// with the result routed by the pair's role (see epilogue.cuh).
//
// Design (one CTA = one 128-row query tile of NT heads that share a kv head):
//   warps 0 .. 4*NT-1  softmax: warpgroup t owns tile t, one thread per row
//                      (TMEM lane), online softmax in the exp2 domain
//   warp 4*NT          TMA producer: Q once, then K_j / V_j tiles into a
//                      2-stage ring (128-byte swizzle, 128 x 64 boxes)
//   warp 4*NT+1        MMA issuer (one thread): S_t = Q_t K_j^T (SMEM x SMEM),
//                      O_t += P_t V_j (P from TMEM, V from SMEM), fp32 in TMEM
// TMEM columns: S_t at 128 t, O_t at 128 (NT + t); P_t (bf16 pairs) overwrites
// the first 64 columns of S_t.  Before S_t(j+1) is written the issuer waits for
// O_t += P_t(j) V_j to complete (the two MMAs have different accumulators, so
// their order is not implied).
// Causal block skip: a tile loads only keys [0, kv_end) where kv_end is the
// last valid row's limit; only tiles past the first row's limit are masked.
// Lazy rescale: the running max moves only when it grows by more than 2^8;
// normalisation by the row sum at the end makes the result exact either way.
//
// Every mbarrier wait is bounded (about 2 s of global time); a wait that gives
// up records CPATTN_ERR_TIMEOUT in a device status word, the CTA drains its
// own copies and MMAs, frees its TMEM and returns without writing output.
#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>
#include <stdlib.h>

#include <mutex>

#include "cpattn_internal.h"
#include "epilogue.cuh"
#include "tmem_ldst.cuh"

namespace cpattn {

__device__ unsigned int g_attn_tc_status;

namespace {

constexpr int kBM = 128;                  // query rows per tile (TMEM lanes)
constexpr int kBN = 128;                  // keys per tile
constexpr int kD = 128;                   // head dim
constexpr int kBoxBytes = 128 * 128;      // 128 rows x 64 bf16 (one swizzle span)
constexpr int kTileBytes = 2 * kBoxBytes; // 128 x 128 bf16
constexpr float kRescaleLog2 = 8.0f;      // lazy-rescale threshold (log2 units)
constexpr unsigned long long kWaitNs = 2000000000ull;

template <int NT>
struct Layout {
  // K and V ring depth: two stages with two query tiles (Q takes 64 KB), three
  // with one (decode tiles stream K/V and want more copies in flight).
  static constexpr int kStages = NT == 2 ? 2 : 3;
  static constexpr int kThreads = (4 * NT + 2) * 32;
  static constexpr int kTmaWarp = 4 * NT;
  static constexpr int kMmaWarp = 4 * NT + 1;
  // TMEM columns: NT == 2: S_0, S_1, O_0, O_1 (128 each).  NT == 1: S buffer
  // 0, O, S buffer 1 (two score tiles, so the next QK product runs while the
  // softmax works on the current one).
  static constexpr int kTmemCols = 512;
  static constexpr int kSBufs = NT == 1 ? 2 : 1;
  static constexpr int q_off = 0;
  static constexpr int k_off = q_off + NT * kTileBytes;
  static constexpr int v_off = k_off + kStages * kTileBytes;
  static constexpr int bar_off = v_off + kStages * kTileBytes;
  // barrier indices
  static constexpr int b_qfull = 0;
  static constexpr int b_qempty = 1;  // the item's last QK MMA is done with Q
  static constexpr int b_kfull = 2;
  static constexpr int b_kempty = b_kfull + kStages;
  static constexpr int b_vfull = b_kempty + kStages;
  static constexpr int b_vempty = b_vfull + kStages;
  static constexpr int b_sfull = b_vempty + kStages;  // per tile, or per score buffer (NT == 1)
  static constexpr int b_pready = b_sfull + NT * kSBufs;
  static constexpr int b_pvdone = b_pready + NT * kSBufs;
  static constexpr int b_ofree = b_pvdone + NT;  // softmax warps have read O_t
  static constexpr int b_pvstep = b_ofree + NT;  // NT == 1: every PV MMA group done
  static constexpr int b_drain = b_pvstep + 1;
  static constexpr int n_bars = b_drain + 1;
  static constexpr int tmem_slot_off = bar_off + n_bars * 8;
  static constexpr int abort_off = tmem_slot_off + 4;
  static constexpr int bytes = abort_off + 4;
  static constexpr int alloc_bytes = bytes + 1024;  // room to align the base to 1024
};

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait for the phase with the given parity.  Returns false if the
// CTA's abort flag is raised (when honour_abort) or the time limit passes; a
// timeout raises the abort flag and records the device status.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                         bool honour_abort = true) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0u) {
      if (honour_abort && *abort_flag) return false;
      if (global_ns() - t0 > kWaitNs) {
        *abort_flag = 1;
        atomicOr(&g_attn_tc_status, 1u);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int c0, int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// D(tmem) (+)= A(smem) * B(smem)
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D(tmem) (+)= A(tmem) * B(smem)
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on `bar` once every tcgen05 operation this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// Instruction descriptor, kind::f16: fp32 accumulate, bf16 A and B.
__host__ __device__ constexpr uint32_t make_idesc(int M, int N, bool b_mn_major) {
  return (1u << 4)                                // D format: f32
         | (1u << 7)                              // A format: bf16
         | (1u << 10)                             // B format: bf16
         | (0u << 15)                             // A K-major
         | ((b_mn_major ? 1u : 0u) << 16)         // B K-major (0) or MN-major (1)
         | ((uint32_t)(N >> 3) << 17)             // N / 8
         | ((uint32_t)(M >> 4) << 24);            // M / 16
}
constexpr uint32_t kIdescQK = make_idesc(kBM, kBN, false);
constexpr uint32_t kIdescPV = make_idesc(kBM, kD, true);

// Shared-memory matrix descriptor, 128-byte swizzle.
__device__ __forceinline__ uint64_t make_sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;   // descriptor version for tcgen05
  d |= (uint64_t)2 << 61;   // SWIZZLE_128B
  return d;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float y;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
  return y;
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&t);
}

// ---------------------------------------------------------------- kernel
// Kernel parameters (three tensor maps and the parameter block) must fit the
// 4 KB kernel-parameter space.
static_assert(sizeof(AttnParams) + 3 * sizeof(CUtensorMap) <= 4096, "kernel parameters too large");

template <int NT, bool kStrictOrder, bool kPersistent, bool kRowPair>
__global__ void __launch_bounds__(Layout<NT>::kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ AttnParams p) {
  using L = Layout<NT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int idx) -> uint32_t { return sb + L::bar_off + 8 * idx; };
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::abort_off);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const PairDesc *pairs = p.pair_table != nullptr ? p.pair_table : p.pairs;
  const int n_pairs = p.pair_table != nullptr ? p.n_table : p.n_pairs;
  const int G = NT == 1 ? p.pack_g : 0;  // query heads per tile in packed mode, else 0
  static_assert(!kRowPair || NT == 2, "row pairs need two tiles per CTA");
  constexpr bool RP = kRowPair;  // tiles = two row blocks of one head
  // Work items handled by this CTA: blockIdx.x, + stride, ... (one item when
  // the grid has a CTA per item; a loop in a persistent launch).
  // A non-persistent launch runs exactly one item per CTA, which the compiler
  // sees (kPersistent false), so no state is carried between items.
  const int stride = kPersistent ? (int)gridDim.x : p.total_ctas;

  // ---- setup (once per CTA)
  if (threadIdx.x == 0) {
    mbar_init(bar(L::b_qfull), 1);
    mbar_init(bar(L::b_qempty), 1);
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(bar(L::b_kfull + s), 1);
      mbar_init(bar(L::b_kempty + s), 1);
      mbar_init(bar(L::b_vfull + s), 1);
      mbar_init(bar(L::b_vempty + s), 1);
    }
    for (int t = 0; t < NT * L::kSBufs; ++t) {
      mbar_init(bar(L::b_sfull + t), 1);
      mbar_init(bar(L::b_pready + t), 4);
    }
    for (int t = 0; t < NT; ++t) {
      mbar_init(bar(L::b_pvdone + t), 1);
      mbar_init(bar(L::b_ofree + t), 4);
    }
    mbar_init(bar(L::b_pvstep), 1);
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
    tmem_alloc(sb + L::tmem_slot_off, L::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + L::tmem_slot_off);

  // ---- work item geometry (every role decodes the same items identically)
  //   per-head tiles (pack_g == 0): (pair, query rows, heads, batch) -- 128
  //     rows of a pair of heads, or 256 rows of one head with row pairs
  //   packed decode tiles (pack_g > 0, NT == 1): (pair, kv split, kv head, batch)
  struct Item {
    const PairDesc *pd;
    int h0, hk, i0, q_rows, split, b, qt, n_kv, n_unmasked;
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
    it.split = 0;
    it.ks = 0;
    it.ke = pd.kv_len;
    if (G == 0) {
      // Tile t of the item: head h0 + t (two heads of a group) or, with row
      // pairs, rows 128 t .. of the item's 256 rows of head h0.
      const int hpi = RP ? 1 : NT, rpi = RP ? 2 * kBM : kBM;
      const int n_hg = p.Hq / hpi;
      const int hg = local % n_hg;
      local /= n_hg;
      it.qt = pd.n_qtiles - 1 - local / p.B;  // longest tiles first
      it.h0 = hg * hpi;
      it.hk = it.h0 / (p.Hq / p.Hkv);
      it.i0 = it.qt * rpi;
      it.q_rows = min(rpi, pd.q_len - it.i0);
    } else {
      it.hk = local % p.Hkv;
      local /= p.Hkv;
      it.split = local / p.B;
      it.qt = 0;
      it.h0 = it.hk * G;
      it.i0 = 0;
      it.q_rows = pd.q_len;
      it.ks = (int64_t)it.split * p.kv_split;
      it.ke = it.ks + p.kv_split < it.ke ? it.ks + p.kv_split : it.ke;
    }
    it.b = local % p.B;
    // Keys [ks, kv_end) are visible to some row of the tile; [ks, full_end) to every row.
    int64_t kv_end = it.ke, full_end = it.ke;
    if (p.causal) {
      const int64_t last_lim = (int64_t)(it.i0 + it.q_rows - 1) + pd.delta + 1;
      const int64_t first_lim = (int64_t)it.i0 + pd.delta + 1;
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
    // K/V loads count up across items (stage g % S, phase g / S); Q of an
    // item waits until the previous item's QK MMAs are done with Q.
    if (lane == 0) {
      int issued_k[L::kStages] = {0}, issued_v[L::kStages] = {0}, issued_q = 0;
      int g = 0, nitem = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < p.total_ctas && ok; item += stride) {
        Item it;
        decode(item, it);
        if (it.n_kv == 0) continue;
        if (nitem > 0 && !wait_bar(bar(L::b_qempty), (nitem - 1) & 1, abort_flag)) { ok = false; break; }
        mbar_expect_tx(bar(L::b_qfull), NT * kTileBytes);
        for (int t = 0; t < NT; ++t)
          for (int half = 0; half < 2; ++half)
            tma_load_4d(sb + L::q_off + t * kTileBytes + half * kBoxBytes, &tm_q, bar(L::b_qfull),
                        half * 64, it.h0 + (RP ? 0 : t), it.pd->q_row0 + it.i0 + (RP ? t * kBM : 0),
                        it.b);  // packed map: heads h0..
        ++issued_q;
        for (int j = 0; j < it.n_kv; ++j, ++g) {
          const int st = g % L::kStages;
          const int kv_row = it.pd->kv_row0 + (int)it.ks + j * kBN;
          if (g >= L::kStages &&
              !wait_bar(bar(L::b_kempty + st), ((g / L::kStages) - 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          mbar_expect_tx(bar(L::b_kfull + st), kTileBytes);
          for (int half = 0; half < 2; ++half)
            tma_load_4d(sb + L::k_off + st * kTileBytes + half * kBoxBytes, &tm_k,
                        bar(L::b_kfull + st), half * 64, it.hk, kv_row, it.b);
          ++issued_k[st];
          if (g >= L::kStages &&
              !wait_bar(bar(L::b_vempty + st), ((g / L::kStages) - 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          mbar_expect_tx(bar(L::b_vfull + st), kTileBytes);
          for (int half = 0; half < 2; ++half)
            tma_load_4d(sb + L::v_off + st * kTileBytes + half * kBoxBytes, &tm_v,
                        bar(L::b_vfull + st), half * 64, it.hk, kv_row, it.b);
          ++issued_v[st];
        }
        ++nitem;
        if constexpr (!kPersistent) break;
      }
      if (!ok) {
        // Let the copies already in flight land before the CTA exits.
        if (issued_q > 0) wait_bar(bar(L::b_qfull), (issued_q - 1) & 1, abort_flag, false);
        for (int s = 0; s < L::kStages; ++s) {
          if (issued_k[s] > 0) wait_bar(bar(L::b_kfull + s), (issued_k[s] - 1) & 1, abort_flag, false);
          if (issued_v[s] > 0) wait_bar(bar(L::b_vfull + s), (issued_v[s] - 1) & 1, abort_flag, false);
        }
      }
    }
    __syncwarp();
  } else if (warp == L::kMmaWarp) {
    // ================================================= MMA issuer (one thread)
    // Issue order per KV step j (ping-pong between the two tiles):
    //   O_0 += P_0(j) V_j,  S_0(j+1) = Q_0 K_{j+1}^T,  O_1 += P_1(j) V_j,  S_1(j+1) = ...
    // While tile 0's softmax turns S_0(j+1) into P_0(j+1), the tensor pipe
    // runs tile 1's two MMAs, and the other way round.
    // S_t(j+1) overwrites the TMEM columns that hold P_t(j), which the PV MMA
    // issued just before reads.  The default schedule relies on the tensor
    // pipe executing one thread's MMAs in issue order (PTX states that order
    // only for MMAs sharing an accumulator); kStrictOrder inserts a wait for
    // the PV MMA to complete before S_t(j+1) is issued.
    // Across items: the first PV of an item (which overwrites O_t) waits until
    // the softmax warps have read the previous item's O_t (ofree_t).
    if (lane == 0) {
      // Descriptors of the first 16-column slice of tile 0 / stage 0 of each
      // operand; other tiles, stages and slices add their byte offset (>> 4)
      // to the start-address field (shared memory stays below 256 KB, so the
      // 14-bit field cannot carry).
      const uint64_t dq0 = make_sdesc(sb + L::q_off, 16, 1024);
      const uint64_t dk0 = make_sdesc(sb + L::k_off, 16, 1024);
      const uint64_t dv0 = make_sdesc(sb + L::v_off, kBoxBytes, 1024);
      constexpr uint64_t kTileStep = kTileBytes >> 4;
      // S (TMEM columns s_col..) = Q_t K^T; O (o_col..) (+)= P V with P in
      // the first 64 columns of the score tile.
      auto issue_qk_at = [&](int t, int st, int s_col) {
        const uint64_t dq = dq0 + (uint64_t)t * kTileStep;
        const uint64_t dk = dk0 + (uint64_t)st * kTileStep;
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint64_t off = (uint64_t)(((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4);
          mma_ss(tmem + s_col, dq + off, dk + off, kIdescQK, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_pv_at = [&](int s_col, int o_col, int st, bool accumulate) {
        const uint64_t dv = dv0 + (uint64_t)st * kTileStep;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          mma_ts(tmem + o_col, tmem + s_col + kk * 8,
                 dv + (uint64_t)((kk * 16 * 128) >> 4), kIdescPV, (accumulate || kk > 0) ? 1u : 0u);
        }
      };
      auto issue_qk = [&](int t, int st) { issue_qk_at(t, st, t * 128); };
      auto issue_pv = [&](int t, int st, bool accumulate) {
        issue_pv_at(t * 128, (NT + t) * 128, st, accumulate);
      };
      bool ok = true;
      int g = 0, nitem = 0;  // KV steps and non-empty items issued so far
      if constexpr (NT == 1) {
        // One tile, two score buffers (step g uses buffer g & 1, at TMEM
        // column 256 * (g & 1)); O at column 128.  QK of step g + 2 reuses
        // the buffer whose P the PV of step g reads, and is issued right after
        // it (in-order tensor pipe; kStrictOrder waits for every PV instead).
        // Every PV commits pvstep: the softmax of step g + 1 may run before
        // the PV of step g completes and must wait for it before rescaling O.
        // (Phase-parity waits stay unambiguous: when the softmax of step g + 1
        // waits, the PV of step g - 1 is complete -- the QK of step g + 1 was
        // issued after it -- and the PV of step g + 1 cannot be.)  pvdone
        // completes once per item, after its last PV.
        auto qk_step = [&](int gk, bool last_qk) -> bool {
          const int sk = gk % L::kStages;
          if (!wait_bar(bar(L::b_kfull + sk), (gk / L::kStages) & 1, abort_flag)) return false;
          tc_fence_after();
          issue_qk_at(0, sk, (gk & 1) * 256);
          mma_commit(bar(L::b_sfull + (gk & 1)));
          mma_commit(bar(L::b_kempty + sk));
          if (kPersistent && last_qk) mma_commit(bar(L::b_qempty));
          return true;
        };
        for (int item = blockIdx.x; item < p.total_ctas && ok; item += stride) {
          Item it;
          decode(item, it);
          const int n_kv = it.n_kv;
          if (n_kv == 0) continue;
          if (!wait_bar(bar(L::b_qfull), nitem & 1, abort_flag)) { ok = false; break; }
          for (int j = 0; j < 2 && j < n_kv && ok; ++j) ok = qk_step(g + j, j == n_kv - 1);
          for (int j = 0; j < n_kv && ok; ++j) {
            const int gj = g + j;
            const int buf = gj & 1;
            const int sv = gj % L::kStages;
            if (!wait_bar(bar(L::b_vfull + sv), (gj / L::kStages) & 1, abort_flag) ||
                !wait_bar(bar(L::b_pready + buf), (gj >> 1) & 1, abort_flag) ||
                (kPersistent && j == 0 && nitem > 0 &&
                 !wait_bar(bar(L::b_ofree), (nitem - 1) & 1, abort_flag))) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_pv_at(buf * 256, 128, sv, j > 0);
            mma_commit(bar(L::b_vempty + sv));
            mma_commit(bar(L::b_pvstep));
            if (j == n_kv - 1) mma_commit(bar(L::b_pvdone));
            if (kStrictOrder && !wait_bar(bar(L::b_pvstep), gj & 1, abort_flag)) {
              ok = false;
              break;
            }
            if (j + 2 < n_kv) ok = qk_step(gj + 2, j + 2 == n_kv - 1);
          }
          g += n_kv;
          ++nitem;
          if constexpr (!kPersistent) break;
        }
      }
      for (int item = blockIdx.x; item < p.total_ctas && ok && NT == 2; item += stride) {
        Item it;
        decode(item, it);
        const int n_kv = it.n_kv;
        if (n_kv == 0) continue;
        if (!wait_bar(bar(L::b_qfull), nitem & 1, abort_flag) ||
            !wait_bar(bar(L::b_kfull + g % L::kStages), (g / L::kStages) & 1, abort_flag)) {
          ok = false;
          break;
        }
        if (kStrictOrder && nitem > 0) {
          // S_t(0) overwrites P_t of the previous item's last PV.
          for (int t = 0; t < NT && ok; ++t)
            ok = wait_bar(bar(L::b_pvdone + t), (g - 1) & 1, abort_flag);
          if (!ok) break;
        }
        tc_fence_after();
        for (int t = 0; t < NT; ++t) {
          issue_qk(t, g % L::kStages);
          mma_commit(bar(L::b_sfull + t));
        }
        mma_commit(bar(L::b_kempty + g % L::kStages));
        if (kPersistent && n_kv == 1) mma_commit(bar(L::b_qempty));
        for (int j = 0; j < n_kv && ok; ++j) {
          const int gj = g + j;
          const int st = gj % L::kStages;
          const int st1 = (gj + 1) % L::kStages;
          const bool more = j + 1 < n_kv;
          for (int t = 0; t < NT && ok; ++t) {
            // Each wait sits right before the first MMA that needs it.
            if ((t == 0 && !wait_bar(bar(L::b_vfull + st), (gj / L::kStages) & 1, abort_flag)) ||
                !wait_bar(bar(L::b_pready + t), gj & 1, abort_flag) ||
                (kPersistent && j == 0 && nitem > 0 &&
                 !wait_bar(bar(L::b_ofree + t), (nitem - 1) & 1, abort_flag))) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_pv(t, st, j > 0);
            if (t == NT - 1) mma_commit(bar(L::b_vempty + st));
            if (kStrictOrder || !more) mma_commit(bar(L::b_pvdone + t));
            if (more) {
              if (t == 0 &&
                  !wait_bar(bar(L::b_kfull + st1), ((gj + 1) / L::kStages) & 1, abort_flag)) {
                ok = false;
                break;
              }
              if (kStrictOrder) {
                if (!wait_bar(bar(L::b_pvdone + t), gj & 1, abort_flag)) { ok = false; break; }
              }
              tc_fence_after();
              issue_qk(t, st1);
              mma_commit(bar(L::b_sfull + t));
              if (t == NT - 1) {
                mma_commit(bar(L::b_kempty + st1));
                if (kPersistent && j + 2 == n_kv) mma_commit(bar(L::b_qempty));  // last QK
              }
            }
          }
        }
        g += n_kv;
        ++nitem;
        if constexpr (!kPersistent) break;
      }
      if (!ok) {
        mma_commit(bar(L::b_drain));
        wait_bar(bar(L::b_drain), 0, abort_flag, false);
      }
    }
    __syncwarp();
  } else {
    // ================================================= softmax warpgroups
    const int t = warp >> 2;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // row in the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t t_s0 = tmem + lane_off + t * 128;  // NT == 1: buffer 0; buffer 1 at + 256
    const uint32_t t_o = tmem + lane_off + (NT + t) * 128;
    const float sl2 = p.scale_log2;
    bool ok = true;
    int g = 0, nitem = 0;
    for (int item = blockIdx.x; item < p.total_ctas && ok; item += stride) {
      Item it;
      decode(item, it);
      const PairDesc &pd = *it.pd;
      const int n_kv = it.n_kv;
      // Query row (inside the pair's chunk) and head of this tile row.
      const int trow = RP ? t * kBM + r : r;  // row within the item
      const int qrow = G == 0 ? it.i0 + trow : r / G;
      const int head = G == 0 ? it.h0 + (RP ? 0 : t) : it.h0 + r % G;
      const bool valid = G == 0 ? trow < it.q_rows : qrow < it.q_rows;
      int64_t lim = it.ke;  // this row's visible keys: [ks, lim)
      if (p.causal) {
        const int64_t c = (int64_t)qrow + pd.delta + 1;
        lim = c < lim ? c : lim;
      }
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = 0; j < n_kv; ++j) {
        // Warp-uniform outcome: the TMEM accesses below are warp-collective.
        // Score buffer of this step and the phase of its barrier.
        const int sbuf = NT == 1 ? ((g + j) & 1) : t;
        const uint32_t sphase = NT == 1 ? (((g + j) >> 1) & 1) : ((g + j) & 1);
        const uint32_t t_s = t_s0 + (NT == 1 ? (uint32_t)((g + j) & 1) * 256u : 0u);
        if (!__all_sync(0xffffffffu, wait_bar(bar(L::b_sfull + sbuf), sphase, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[128];
        tmem_ld_x128(t_s, sr);
        float s[128];
#pragma unroll
        for (int c = 0; c < kBN; ++c) s[c] = __uint_as_float(sr[c]);
        if (j >= it.n_unmasked) {
          int64_t nv = lim - it.ks - (int64_t)j * kBN;
          const int nvis = nv < 0 ? 0 : (nv > kBN ? kBN : (int)nv);
#pragma unroll
          for (int c = 0; c < kBN; ++c)
            if (c >= nvis) s[c] = -INFINITY;
        }
        // Row max: eight independent chains of 3-input maxima (short
        // dependency chains keep the softmax off the MMA critical path).
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
          if (NT == 1) {
            // The previous step's PV may still be accumulating into O.
            if (!__all_sync(0xffffffffu,
                            wait_bar(bar(L::b_pvstep), (g + j - 1) & 1, abort_flag))) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          const float a = rescale_o ? alpha : 1.f;
          if constexpr (kPersistent && NT == 2) {
            // Eight columns at a time, not unrolled: the 128 scores stay live
            // across this rarely taken branch, and in the looping kernel a
            // wider slice of O here pushes the whole loop into spilling
            // registers (measured: 268 -> 36 spilled bytes, +3 % throughput).
#pragma unroll 1
            for (int cc = 0; cc < kD / 8; ++cc) {
              uint32_t ov[8];
              tmem_ld_x8(t_o + cc * 8, ov);
#pragma unroll
              for (int x = 0; x < 8; ++x) ov[x] = __float_as_uint(__uint_as_float(ov[x]) * a);
              tmem_st_x8(t_o + cc * 8, ov);
            }
          } else {
#pragma unroll
            for (int cc = 0; cc < kD / 32; ++cc) {
              uint32_t ov[32];
              tmem_ld_x32(t_o + cc * 32, ov);
#pragma unroll
              for (int x = 0; x < 32; ++x) ov[x] = __float_as_uint(__uint_as_float(ov[x]) * a);
              tmem_st_x32(t_o + cc * 32, ov);
            }
          }
        }
        // p = 2^(s * scale * log2e - m): the scale-and-shift runs two columns per
        // instruction (f32x2 FMA), the row sum in four independent f32x2 chains.
        const float neg_m = m_run == -INFINITY ? 0.f : -m_run;
        const float2 sl2v = make_float2(sl2, sl2);
        const float2 negm = make_float2(neg_m, neg_m);
        float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                         make_float2(0.f, 0.f)};
        // Four quarters of 32 columns: each quarter's P is stored (16 packed
        // columns) as soon as it exists, so few registers stay live.
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
          tmem_st_x16(t_s + qq * 16, pk);
        }
        const float2 a01 = __fadd2_rn(acc[0], acc[1]);
        const float2 a23 = __fadd2_rn(acc[2], acc[3]);
        const float2 a03 = __fadd2_rn(a01, a23);
        l_run += a03.x + a03.y;
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::b_pready + sbuf));
      }
      if (!ok) break;

      // ---- epilogue: O_t / l, LSE, routed by the pair's role
      if (n_kv > 0) {
        // pvdone_t completes once per KV step in the two-tile strict
        // schedule, else once per item.
        const uint32_t par = (kStrictOrder && NT == 2) ? ((g + n_kv - 1) & 1) : (nitem & 1);
        ok = __all_sync(0xffffffffu, wait_bar(bar(L::b_pvdone + t), par, abort_flag));
        tc_fence_after();
        if (!ok) break;
      }
      // One launch for all Pass-KV steps: accumulator updates of a tile row
      // block happen in visit order (progress counter per tile, head, batch).
      int32_t *dep = nullptr;
      if (kPersistent && p.dep_counters != nullptr && G == 0 &&
          (pd.mode == kAccInit || pd.mode == kAccMerge || pd.mode == kAccFinal))
        dep = p.dep_counters + pd.dep_base +
              ((int64_t)(RP ? it.qt * 2 + t : it.qt) * p.Hq + head) * p.B + it.b;
      // Each of the tile's 4 warps adds 1 when its rows are written, so the
      // rows' earlier visits are done once the count reaches 4 * visit.  Every
      // warp waits and publishes for itself: no barrier spans warps whose
      // abort decisions may differ.
      if (dep != nullptr && pd.visit > 0) {
        int got = 1;
        if (lane == 0) {
          const int target = 4 * pd.visit + p.dep_hold;
          const unsigned long long t0 = global_ns();
          for (uint32_t spin = 0;; ++spin) {
            int v;
            asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(dep) : "memory");
            if (v >= target) break;
            if ((spin & 63u) == 63u && (*abort_flag || global_ns() - t0 > kWaitNs)) {
              *abort_flag = 1;
              atomicOr(&g_attn_tc_status, 1u);
              got = 0;
              break;
            }
          }
        }
        __syncwarp();
        if (!__shfl_sync(0xffffffffu, got, 0)) { ok = false; break; }
      }
      const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
      const float lse = l_run > 0.f ? (m_run + log2f(l_run)) * 0.6931471805599453f : -INFINITY;
      RowSink sink;
      if (valid) sink.init(p, pd, it.b, head, qrow, lse, true, G == 0 ? -1 : pd.slot + it.split);
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
      if (kPersistent && n_kv > 0) {
        // O_t has been read: the next item's first PV may overwrite it.
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::b_ofree + t));
      }
      if (dep != nullptr && pd.mode != kAccFinal) {
        __syncwarp();
        if (lane == 0) {
          __threadfence();
          asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(dep) : "memory");
        }
      }
      g += n_kv;
      if (n_kv > 0) ++nitem;
      if constexpr (!kPersistent) break;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == L::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  // Looked up once (function-local static: initialised by one thread).
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
              int64_t sb, int64_t ss, int64_t sh, uint32_t box_h = 1, uint32_t box_s = 128) {
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

template <int NT, bool kStrictOrder, bool kPersistent, bool kRowPair>
cudaError_t launch_nt(AttnParams &p, cudaStream_t stream) {
  using L = Layout<NT>;
  int total = 0;
  if (p.pair_table != nullptr) {
    // Device-resident table: the caller computed cta_begin / n_qtiles and the total.
    total = p.total_ctas;
  }
  for (int x = 0; x < (p.pair_table != nullptr ? 0 : p.n_pairs); ++x) {
    PairDesc &pd = p.pairs[x];
    if (p.pack_g > 0) {  // n_qtiles counts kv splits in packed mode
      pd.n_qtiles = (pd.kv_len + p.kv_split - 1) / p.kv_split;
      pd.cta_begin = total;
      total += pd.n_qtiles * p.Hkv * p.B;
    } else {
      const TcItemShape sh = attn_tc_item_shape(p);
      pd.n_qtiles = (pd.q_len + sh.rows - 1) / sh.rows;
      pd.cta_begin = total;
      total += pd.n_qtiles * (p.Hq / sh.heads) * p.B;
    }
  }
  if (p.pair_table == nullptr) p.total_ctas = total;
  if (total == 0) return cudaSuccess;
  CUtensorMap mq, mk, mv;
  const uint32_t qbox_h = p.pack_g > 0 ? (uint32_t)p.pack_g : 1u;
  const uint32_t qbox_s = p.pack_g > 0 ? (uint32_t)(kBM / p.pack_g) : (uint32_t)kBM;
  if (!make_map(&mq, p.q, p.B, p.q_rows_total, p.Hq, kD, p.q_sb, p.q_ss, p.q_sh, qbox_h, qbox_s) ||
      !make_map(&mk, p.k, p.B, p.kv_rows_total, p.Hkv, kD, p.k_sb, p.k_ss, p.k_sh) ||
      !make_map(&mv, p.v, p.B, p.kv_rows_total, p.Hkv, kD, p.v_sb, p.v_ss, p.v_sh))
    return cudaErrorInvalidValue;
  // Per device: the shared-memory attribute of this instantiation, set once,
  // and the SM count (host threads may launch on several devices at once).
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
      cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<NT, kStrictOrder, kPersistent, kRowPair>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           L::alloc_bytes);
      if (e != cudaSuccess) return e;
      e = cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return e;
      configured[dev] = true;
    }
    sm_count = sms[dev];
  }
  // Persistent launch: one CTA per SM (shared memory admits only one), each
  // looping over work items; otherwise one CTA per item.
  int grid = total;
  if (p.persistent_ctas > 0) {
    p.persistent_ctas = sm_count < total ? sm_count : total;
    grid = p.persistent_ctas;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(L::kThreads);
  cfg.dynamicSmemBytes = L::alloc_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if (p.dep_counters != nullptr) {
    // CTAs wait on other CTAs' progress counters: they must all be resident.
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, attn_tc_kernel<NT, kStrictOrder, kPersistent, kRowPair>, mq, mk,
                            mv, p);
}

}  // namespace

bool attn_tc_supported(const AttnParams &p) {
  if (p.in_f32 || p.D != kD || p.q_rows_total <= 0 || p.kv_rows_total <= 0) return false;
  if (p.pack_g > 0) {
    // Packed decode tiles: the group fills whole TMA boxes and every query
    // row of a pair fits in one 128-row tile; splits are whole KV tiles.
    if (p.pack_g != p.Hq / p.Hkv || kBM % p.pack_g != 0 || p.kv_split <= 0 || p.kv_split % kBN)
      return false;
    for (int x = 0; x < p.n_pairs; ++x)
      if (p.pairs[x].q_len > kBM / p.pack_g) return false;
  }
  return true;
}

// CPATTN_STRICT_MMA_ORDER=1 selects the schedule that waits for each PV MMA
// to complete before the next QK MMA overwrites P (see the MMA issuer).
bool strict_mma_order() {
  const char *e = getenv("CPATTN_STRICT_MMA_ORDER");
  return e != nullptr && e[0] != '\0' && e[0] != '0';
}

TcItemShape attn_tc_item_shape(const AttnParams &p) {
  if (p.pack_g > 0) return {kBM, 1};
  return (p.Hq / p.Hkv) % 2 == 0 ? TcItemShape{kBM, 2} : TcItemShape{2 * kBM, 1};
}

template <int NT, bool kRowPair>
cudaError_t launch_nt_any(AttnParams &p, cudaStream_t stream, bool strict) {
  const bool pers = p.persistent_ctas > 0;
  if (strict)
    return pers ? launch_nt<NT, true, true, kRowPair>(p, stream)
                : launch_nt<NT, true, false, kRowPair>(p, stream);
  return pers ? launch_nt<NT, false, true, kRowPair>(p, stream)
              : launch_nt<NT, false, false, kRowPair>(p, stream);
}

cudaError_t launch_attn_tc(AttnParams &p, cudaStream_t stream) {
  const bool strict = strict_mma_order();
  // Per-head tiles always pair two 128-row tiles in a CTA (two heads of a
  // group, or two row blocks of one head); packed decode tiles run alone.
  p.row_pair = (p.pack_g == 0 && (p.Hq / p.Hkv) % 2 != 0) ? 1 : 0;
  if (p.pack_g != 0) return launch_nt_any<1, false>(p, stream, strict);
  return p.row_pair ? launch_nt_any<2, true>(p, stream, strict)
                    : launch_nt_any<2, false>(p, stream, strict);
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
