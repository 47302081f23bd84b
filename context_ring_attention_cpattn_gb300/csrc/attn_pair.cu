// Partial attention of (Q-chunk, KV-chunk) pairs on a pair of SMs of sm_103a
// (tcgen05 with cta_group::2, TMEM, TMA), bf16 inputs, head_dim 128.
//
// What one pair computes: the per-rank step of context-parallel ring
// attention ("Scaling LLM Inference ...", techreport rewrite, section
// "Context Parallelism for Million-Token Contexts", Pass-KV / Pass-Q bullets;
// the pages name only "a fast attention kernel" and give no design):
//   s_ij = scale * q_i . k_j  for keys with kv_pos(j) <= q_pos(i) (causal),
//   LSE_i = log sum_j exp(s_ij),  O_i = sum_j exp(s_ij - LSE_i) v_j,
// with the result routed by the pair's role (epilogue.cuh).
//
// Design.  A cluster of two CTAs (a CTA pair on two SMs) owns one 256-row
// work item: the same 128 query rows of two heads that share a kv head, or
// two consecutive 128-row blocks of one head (odd GQA groups); CTA r holds
// tile r.  One thread of CTA 0 issues every MMA as an M = 256 tcgen05.mma
// that spans both SMs: A rows (queries) and accumulator lanes come from each
// CTA's own shared memory and TMEM, the B operand is split between the two
// CTAs -- CTA r loads keys 64r..64r+63 of each 128-key K tile and head-dim
// columns 64r..64r+63 of each V tile -- so each SM reads half of every K/V
// tile from L2 and from its shared memory.
//   S(j)  = Q K_j^T   (A, B in shared memory)      into score buffer j % 2
//   O    += P(j) V_j  (A = P from TMEM, B in SMEM) into O
// TMEM (512 columns per CTA): score buffers at 0 and 128, O at 256, P buffers
// (bf16 pairs) at 384 and 448.  Every TMEM region an MMA reads or writes is
// free by construction when the MMA is issued, and no ordering between MMAs
// of different accumulators is assumed:
//   - S(j + 2) is issued once the softmax of step j has loaded S(j) into
//     registers (it signals "score buffer free"), ahead of PV(j), so a warp's
//     next scores are ready when it finishes a step;
//   - the softmax writes P(j + 2) into P buffer j % 2 only after PV(j), which
//     read it, is complete (PV(j)'s commit also releases its K/V stage);
//   - O is rescaled only after the previous step's PV is complete, and the
//     next PV waits for the P that the rescaling warp publishes afterwards.
//
// Warp roles per CTA: 8 softmax warps, one TMA producer warp, one MMA warp
// (CTA 0: issues the MMAs; CTA 1: a relay that forwards the completion of
// this CTA's loads to CTA 0's barriers).  Softmax warp w reads TMEM lanes
// 32 (w % 4) .. and takes the KV steps of parity w / 4, all 128 keys of each:
// the two warps of a row run a step apart, so one's waits overlap the
// other's arithmetic.  Online softmax in the exp2 domain with one lazy
// reference maximum per row shared by the two warps and decided in step
// order (it moves only when a step's maximum exceeds it by more than 2^8).
// Causal block skip: an item loads only keys below its last row's limit;
// only tiles past its first row's limit are masked.
//
// Measured on GB300 (one 8192 x 8192 causal pair, 16/1 heads, per 128-key
// step of a CTA pair; tcgen05 alone runs an M = 256 MMA in 64 cycles):
// a cluster-scope release on each signal cost ~1300 cycles, a single
// divergent lane issuing MMAs ~60 cycles per MMA, and two warps splitting a
// step's keys stalled together on every wait; the structure above avoids all
// three.
//
// Every wait is bounded (AttnParams::wait_ns of global time); a wait that
// gives up records CPATTN_ERR_TIMEOUT in a device status word and raises the
// abort flag of both CTAs; each CTA then lets its own copies and MMAs land,
// frees its TMEM and returns without writing output.
#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>

#include <mutex>

#include "cpattn_internal.h"
#include "epilogue.cuh"
#include "tc_ptx.cuh"
#include "tmem_ldst.cuh"

namespace cpattn {

__device__ unsigned int g_attn_pair_status;

namespace {

using namespace tc;

constexpr int kRows = 128;               // query rows per CTA (TMEM lanes)
constexpr int kKeys = 128;               // keys per KV step
constexpr int kD = 128;                  // head dim
constexpr int kStages = 5;               // K and V ring depth
constexpr float kRescaleLog2 = 8.0f;     // lazy-rescale threshold (log2 units)
constexpr unsigned long long kDrainNs = 20000000ull;  // abort path: wait for own copies

struct PairLayout {
  // Softmax warps: two per 32-row quad (warp w reads TMEM lanes 32 (w % 4) ..),
  // taking alternate KV steps: warp w handles the steps j with j % 2 == w / 4.
  static constexpr int kSoftmaxWarps = 8;
  static constexpr int kTmaWarp = kSoftmaxWarps;
  static constexpr int kMmaWarp = kSoftmaxWarps + 1;
  static constexpr int kThreads = (kSoftmaxWarps + 2) * 32;
  // Shared memory (1024-byte aligned base; every tile 1024-aligned for the
  // 128-byte swizzle).
  static constexpr int q_box = kRows * 128;     // 128 rows x 64 bf16
  static constexpr int q_bytes = 2 * q_box;
  static constexpr int k_box = 64 * 128;        // 64 keys x 64 bf16
  static constexpr int k_bytes = 2 * k_box;     // this CTA's 64 keys x 128 d
  static constexpr int v_bytes = kKeys * 128;   // 128 keys x this CTA's 64 d
  static constexpr int q_off = 0;
  static constexpr int k_off = q_off + q_bytes;
  static constexpr int v_off = k_off + kStages * k_bytes;
  static constexpr int bar_off = v_off + kStages * v_bytes;
  // barrier indices
  static constexpr int b_qfull = 0;
  static constexpr int b_qempty = 1;
  static constexpr int b_kfull = 2;
  static constexpr int b_vfull = b_kfull + kStages;
  static constexpr int b_kvempty = b_vfull + kStages;  // K and V of a stage are consumed
  static constexpr int b_sfull = b_kvempty + kStages;  // per score buffer
  static constexpr int b_sfree = b_sfull + 2;          // per score buffer: loaded by the softmax (CTA 0's)
  static constexpr int b_pready = b_sfree + 2;         // per P buffer (CTA 0's are used)
  static constexpr int b_ofull = b_pready + 2;         // an item's last PV
  static constexpr int b_ofree = b_ofull + 1;          // softmax warps have read O (CTA 0's)
  static constexpr int b_dec = b_ofree + 1;            // per row quad: a step's reference decided
  static constexpr int b_xsum = b_dec + 4;             // per row quad: both warps' sums posted
  static constexpr int b_drain = b_xsum + 4;
  static constexpr int n_bars = b_drain + 1;
  static constexpr int mref_off = bar_off + n_bars * 8;  // f32 [128]: a row's reference maximum
  static constexpr int xsum_off = mref_off + kRows * 4;  // f32 [2][128]: each warp's row sum
  static constexpr int xm_off = xsum_off + 2 * kRows * 4;  // f32 [2][128]: ... and its reference
  static constexpr int tmem_slot_off = xm_off + 2 * kRows * 4;
  static constexpr int abort_off = tmem_slot_off + 4;
  static constexpr int bytes = abort_off + 4;
  static constexpr int alloc_bytes = bytes + 1024;
  // TMEM columns
  static constexpr int t_s = 0;    // score buffers at 0 and 128
  static constexpr int t_o = 256;  // O
  static constexpr int t_p = 384;  // P buffers at 384 and 448
  static constexpr int kTmemCols = 512;
};

constexpr uint32_t kIdescQK = make_idesc(2 * kRows, kKeys, false);
constexpr uint32_t kIdescPV = make_idesc(2 * kRows, kD, true);

static_assert(sizeof(AttnParams) + 3 * sizeof(CUtensorMap) <= 4096, "kernel parameters too large");

template <bool kPersistent, bool kRowPair, bool kSegs>
__global__ void __launch_bounds__(PairLayout::kThreads, 1)
    attn_pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ AttnParams p) {
  using L = PairLayout;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int idx) -> uint32_t { return sb + L::bar_off + 8 * idx; };
  const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs
  auto peer_bar = [&](int idx) -> uint32_t { return mapa(bar(idx), rank ^ 1u); };
  auto lead_bar = [&](int idx) -> uint32_t { return rank == 0 ? bar(idx) : mapa(bar(idx), 0); };
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::abort_off);
  const uint32_t peer_abort = mapa(sb + L::abort_off, rank ^ 1u);
  const unsigned long long wait_ns = p.wait_ns;
  auto wait = [&](uint32_t b, uint32_t parity) -> bool {
    return wait_phase<false>(b, parity, abort_flag, &g_attn_pair_status, wait_ns, true, peer_abort);
  };
  auto drain_wait = [&](uint32_t b, uint32_t parity) -> bool {
    return wait_phase<false>(b, parity, abort_flag, &g_attn_pair_status, kDrainNs, false, 0);
  };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const PairDesc *pairs = p.pair_table != nullptr ? p.pair_table : p.pairs;
  const int n_pairs = p.pair_table != nullptr ? p.n_table : p.n_pairs;
  const int cluster = (int)(blockIdx.x >> 1);
  const int stride = kPersistent ? (int)(gridDim.x >> 1) : p.total_ctas;

  // ---- setup
  if (threadIdx.x == 0) {
    const uint32_t full_count = rank == 0 ? 2u : 1u;  // CTA 0: own copies + the relay
    mbar_init(bar(L::b_qfull), full_count);
    mbar_init(bar(L::b_qempty), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(L::b_kfull + s), full_count);
      mbar_init(bar(L::b_vfull + s), full_count);
      mbar_init(bar(L::b_kvempty + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(L::b_sfull + b), 1);
      mbar_init(bar(L::b_sfree + b), 2 * 4);   // the step's four warps in each CTA
      mbar_init(bar(L::b_pready + b), 2 * 4);
    }
    mbar_init(bar(L::b_ofull), 1);
    mbar_init(bar(L::b_ofree), 2 * L::kSoftmaxWarps);
    for (int qd = 0; qd < 4; ++qd) {
      mbar_init(bar(L::b_dec + qd), 1);
      mbar_init(bar(L::b_xsum + qd), 2);
    }
    mbar_init(bar(L::b_drain), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == L::kTmaWarp && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == L::kMmaWarp) {
    tmem_alloc_2(sb + L::tmem_slot_off, L::kTmemCols);
    tmem_relinquish_2();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any remote arrive
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + L::tmem_slot_off);

  // ---- work item geometry (every role of both CTAs decodes items identically)
  // A work item's K/V steps are those of its segments, in order: one pair,
  // or, when the table groups pairs (p.seg_groups), every pair of one query
  // piece in ring order, whose K/V pieces then stream through one on-chip
  // accumulator.  In a group, segment x carries visit = x and slot = the
  // group's size, and all share cta_begin.
  struct Seg {
    int n_kv, n_unmasked;
  };
  // 128-key steps of segment `sp` for query rows i0 .. i0 + q_rows - 1 of its
  // piece: keys [0, kv_end) are visible to some row, [0, full_end) to all.
  auto seg_steps = [&](const PairDesc &sp, int i0, int q_rows) -> Seg {
    int64_t kv_end = sp.kv_len, full_end = sp.kv_len;
    if (p.causal) {
      const int64_t last_lim = (int64_t)(i0 + q_rows - 1) + sp.delta + 1;
      const int64_t first_lim = (int64_t)i0 + sp.delta + 1;
      kv_end = last_lim < kv_end ? last_lim : kv_end;
      full_end = first_lim < full_end ? first_lim : full_end;
    }
    if (kv_end < 0) kv_end = 0;
    if (full_end < 0) full_end = 0;
    return {(int)((kv_end + kKeys - 1) / kKeys), (int)(full_end / kKeys)};
  };
  struct Item {
    const PairDesc *pd;  // first segment
    int n_segs, h0, hk, i0, q_rows, qt, b, n_kv, n_unmasked;  // n_unmasked: one-pair items
  };
  auto decode = [&](int item, Item &it) {
    int lo = 0, hi = n_pairs - 1;  // last pair whose cta_begin <= item
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pairs[mid].cta_begin <= item) lo = mid; else hi = mid - 1;
    }
    if constexpr (kSegs) lo -= pairs[lo].visit;
    const PairDesc &pd = pairs[lo];
    it.pd = &pd;
    it.n_segs = kSegs ? pd.slot : 1;
    int local = item - pd.cta_begin;
    constexpr int hpi = kRowPair ? 1 : 2, rpi = kRowPair ? 2 * kRows : kRows;
    const int n_hg = p.Hq / hpi;
    const int hg = local % n_hg;
    local /= n_hg;
    it.qt = pd.n_qtiles - 1 - local / p.B;  // longest tiles first
    it.b = local % p.B;
    it.h0 = hg * hpi;
    it.hk = it.h0 / (p.Hq / p.Hkv);
    it.i0 = it.qt * rpi;
    it.q_rows = min(rpi, pd.q_len - it.i0);
    if constexpr (kSegs) {
      it.n_kv = 0;
      for (int x = 0; x < it.n_segs; ++x) it.n_kv += seg_steps(it.pd[x], it.i0, it.q_rows).n_kv;
      it.n_unmasked = 0;
    } else {
      const Seg q = seg_steps(pd, it.i0, it.q_rows);
      it.n_kv = q.n_kv;
      it.n_unmasked = q.n_unmasked;
    }
  };
  // Position in an item's step sequence: segment, step within it.
  struct Cursor {
    const PairDesc *sp;
    int left, js, n_kv, n_unmasked;
  };
  auto cursor_at = [&](const Item &it, int j) -> Cursor {
    Cursor c;
    c.sp = it.pd;
    c.left = it.n_segs;
    c.js = j;
    Seg q = seg_steps(*c.sp, it.i0, it.q_rows);
    c.n_kv = q.n_kv;
    c.n_unmasked = q.n_unmasked;
    while (c.js >= c.n_kv && c.left > 1) {
      c.js -= c.n_kv;
      ++c.sp;
      --c.left;
      q = seg_steps(*c.sp, it.i0, it.q_rows);
      c.n_kv = q.n_kv;
      c.n_unmasked = q.n_unmasked;
    }
    return c;
  };
  auto cursor_advance = [&](const Item &it, Cursor &c, int by) {
    c.js += by;
    while (c.js >= c.n_kv && c.left > 1) {
      c.js -= c.n_kv;
      ++c.sp;
      --c.left;
      const Seg q = seg_steps(*c.sp, it.i0, it.q_rows);
      c.n_kv = q.n_kv;
      c.n_unmasked = q.n_unmasked;
    }
  };

  if (warp == L::kTmaWarp) {
    // ================================================= TMA producer (both CTAs)
    // Loads in the order the MMA thread consumes them: Q, K_0, K_1, V_0, K_2,
    // V_1, ..., V_{n-1}; K/V steps count up across items (stage g % kStages,
    // phase g / kStages).  A stage is refilled once the PV MMA of the step
    // that last used it is complete (its QK MMA was issued before it).
    if (lane == 0) {
      int nk[kStages] = {0}, nv[kStages] = {0}, nq = 0;  // loads issued per barrier
      int g = 0, nitem = 0;
      bool ok = true;
      for (int item = cluster; item < p.total_ctas && ok; item += stride) {
        Item it;
        decode(item, it);
        if (it.n_kv == 0) continue;
        if (kPersistent && nitem > 0 && !wait(bar(L::b_qempty), (nitem - 1) & 1)) { ok = false; break; }
        mbar_expect_tx(bar(L::b_qfull), L::q_bytes);
        const int head = it.h0 + (kRowPair ? 0 : (int)rank);
        const int qrow = it.pd->q_row0 + it.i0 + (kRowPair ? (int)rank * kRows : 0);
        // Both 64-column halves of the tile in one copy (the map's third
        // dimension is the half).
        tma_load_5d(sb + L::q_off, &tm_q, bar(L::b_qfull), 0, qrow, 0, head, it.b);
        ++nq;
        // K/V rows of step j: a one-pair item indexes its pair; an item of
        // grouped pairs walks them with cursors (K runs one step ahead of V).
        [[maybe_unused]] Cursor ck, cv;
        if constexpr (kSegs) ck = cv = cursor_at(it, 0);
        auto tile_row = [&](Cursor &c, int j) -> int {
          if constexpr (kSegs) {
            const int row = c.sp->kv_row0 + c.js * kKeys;
            cursor_advance(it, c, 1);
            return row;
          } else {
            return it.pd->kv_row0 + j * kKeys;
          }
        };
        auto load_k = [&](int j) -> bool {
          const int gj = g + j, st = gj % kStages;
          if (gj >= kStages && !wait(bar(L::b_kvempty + st), ((gj / kStages) - 1) & 1)) return false;
          mbar_expect_tx(bar(L::b_kfull + st), L::k_bytes);
          const int row = tile_row(ck, j) + (int)rank * 64;
          tma_load_5d(sb + L::k_off + st * L::k_bytes, &tm_k, bar(L::b_kfull + st), 0, row, 0, it.hk,
                      it.b);
          ++nk[st];
          return true;
        };
        auto load_v = [&](int j) -> bool {
          const int gj = g + j, st = gj % kStages;
          // K_j of this stage waited for the same release (the phase is
          // complete, so this returns at once).
          if (gj >= kStages && !wait(bar(L::b_kvempty + st), ((gj / kStages) - 1) & 1)) return false;
          mbar_expect_tx(bar(L::b_vfull + st), L::v_bytes);
          tma_load_4d(sb + L::v_off + st * L::v_bytes, &tm_v, bar(L::b_vfull + st), (int)rank * 64,
                      it.hk, tile_row(cv, j), it.b);
          ++nv[st];
          return true;
        };
        for (int j = 0; j < it.n_kv && ok; ++j) ok = load_k(j) && (j == 0 || load_v(j - 1));
        if (ok) ok = load_v(it.n_kv - 1);
        g += it.n_kv;
        ++nitem;
        if constexpr (!kPersistent) break;
      }
      if (ok) {
        // Every release the MMA thread sent this CTA has landed before the
        // CTA moves on (CTA 0's commits arrive on CTA 1's barriers).
        for (int s = 0; s < kStages && ok; ++s)
          if (nv[s] > 0) ok = wait(bar(L::b_kvempty + s), (nv[s] - 1) & 1);
        if (ok && kPersistent && nq > 0) ok = wait(bar(L::b_qempty), (nq - 1) & 1);
      } else {
        // Let this CTA's copies in flight land before it exits (on CTA 0 a
        // phase also needs the relay's arrival, so this may run to its bound).
        if (nq > 0) drain_wait(bar(L::b_qfull), (nq - 1) & 1);
        for (int s = 0; s < kStages; ++s) {
          if (nk[s] > 0) drain_wait(bar(L::b_kfull + s), (nk[s] - 1) & 1);
          if (nv[s] > 0) drain_wait(bar(L::b_vfull + s), (nv[s] - 1) & 1);
        }
      }
    }
    __syncwarp();
  } else if (warp == L::kMmaWarp && rank != 0) {
    // ================================================= relay (CTA 1)
    // CTA 0's MMAs read this CTA's tiles: forward each completed load to the
    // matching barrier of CTA 0, in the producer's order.
    if (lane == 0) {
      int g = 0, nitem = 0;
      bool ok = true;
      for (int item = cluster; item < p.total_ctas && ok; item += stride) {
        Item it;
        decode(item, it);
        if (it.n_kv == 0) continue;
        if (!wait(bar(L::b_qfull), nitem & 1)) { ok = false; break; }
        mbar_arrive_cluster(lead_bar(L::b_qfull));
        auto fwd = [&](int base, int j) -> bool {
          const int gj = g + j, st = gj % kStages;
          if (!wait(bar(base + st), (gj / kStages) & 1)) return false;
          mbar_arrive_cluster(lead_bar(base + st));
          return true;
        };
        for (int j = 0; j < it.n_kv && ok; ++j) ok = fwd(L::b_kfull, j) && (j == 0 || fwd(L::b_vfull, j - 1));
        if (ok) ok = fwd(L::b_vfull, it.n_kv - 1);
        g += it.n_kv;
        ++nitem;
        if constexpr (!kPersistent) break;
      }
    }
    __syncwarp();
  } else if (warp == L::kMmaWarp) {
    // ================================================= MMA issuer (CTA 0)
    // Per item: S(0), S(1), then for every step j: S(j + 2), O += P(j) V_j.
    // The whole warp runs the loop, so descriptors and addresses are
    // warp-uniform values; one elected lane issues each group of MMAs and its
    // commits (a single divergent lane issuing spent tens of cycles per MMA
    // outside the tensor pipe).  Every commit goes to both CTAs' barriers.
    // Commits are few (a commit costs tensor-pipe time): per step one after
    // the QK group (score buffer full) and one after the PV group (the K/V
    // stage and the P buffer are free); per item one after the last PV.
    {
      const uint64_t dq0 = make_sdesc(sb + L::q_off, 16, 1024);
      const uint64_t dk0 = make_sdesc(sb + L::k_off, 16, 1024);
      const uint64_t dv0 = make_sdesc(sb + L::v_off, 16, 1024);
      const uint32_t peer_bar0 = peer_bar(0);  // the peer's barriers, same layout
      auto commit_both = [&](int idx) {
        mma_commit_2(bar(idx));
        mma_commit_2(peer_bar0 + 8 * idx);
      };
      auto wait_w = [&](uint32_t b, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu, wait(b, parity));
      };
      bool ok = true;
      int g = 0, nitem = 0;
      for (int item = cluster; item < p.total_ctas && ok; item += stride) {
        Item it;
        decode(item, it);
        const int n_kv = it.n_kv;
        if (n_kv == 0) continue;
        auto issue_qk = [&](int j) -> bool {
          const int gk = g + j, st = gk % kStages;
          // The score buffer is free once its previous step's softmax loaded it.
          if ((gk >= 2 && !wait_w(bar(L::b_sfree + (gk & 1)), ((gk - 2) >> 1) & 1)) ||
              !wait_w(bar(L::b_kfull + st), (gk / kStages) & 1))
            return false;
          tc_fence_after();
          const uint64_t dk = dk0 + (uint64_t)((st * L::k_bytes) >> 4);
          const uint32_t d_s = tmem + L::t_s + (gk & 1) * 128;
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk) {
              const uint64_t qo = (uint64_t)(((kk >> 2) * L::q_box + (kk & 3) * 32) >> 4);
              const uint64_t ko = (uint64_t)(((kk >> 2) * L::k_box + (kk & 3) * 32) >> 4);
              mma_ss_2(d_s, dq0 + qo, dk + ko, kIdescQK, kk > 0 ? 1u : 0u);
            }
            commit_both(L::b_sfull + (gk & 1));
            if (kPersistent && j == n_kv - 1) commit_both(L::b_qempty);  // the item's last QK
          }
          __syncwarp();
          return true;
        };
        if (!wait_w(bar(L::b_qfull), nitem & 1)) { ok = false; break; }
        ok = issue_qk(0) && (n_kv < 2 || issue_qk(1));
        for (int j = 0; j < n_kv && ok; ++j) {
          // S(j + 2) as soon as the softmax of step j has loaded S(j), ahead
          // of PV(j): a warp's next scores are then ready when it needs them.
          if (j + 2 < n_kv && !(ok = issue_qk(j + 2))) break;
          const int gj = g + j, sv = gj % kStages;
          if (!wait_w(bar(L::b_vfull + sv), (gj / kStages) & 1) ||
              !wait_w(bar(L::b_pready + (gj & 1)), (gj >> 1) & 1) ||
              (kPersistent && j == 0 && nitem > 0 && !wait_w(bar(L::b_ofree), (nitem - 1) & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t dv = dv0 + (uint64_t)((sv * L::v_bytes) >> 4);
          const uint32_t a_p = tmem + L::t_p + (gj & 1) * 64;
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < kKeys / 16; ++kk)
              mma_ts_2(tmem + L::t_o, a_p + kk * 8, dv + (uint64_t)((kk * 16 * 128) >> 4), kIdescPV,
                       (j > 0 || kk > 0) ? 1u : 0u);
            commit_both(L::b_kvempty + sv);  // also tells the softmax that P buffer gj % 2 was read
            if (j + 1 == n_kv) commit_both(L::b_ofull);
          }
          __syncwarp();
        }
        g += n_kv;
        ++nitem;
        if constexpr (!kPersistent) break;
      }
      // The softmax warps' last release of O (persistent launches) has landed.
      if (ok && kPersistent && nitem > 0) ok = wait_w(bar(L::b_ofree), (nitem - 1) & 1);
      if (!ok) {
        if (elect_one()) {
          mma_commit_2(bar(L::b_drain));
          drain_wait(bar(L::b_drain), 0);
        }
      }
    }
    __syncwarp();
  } else {
    // ================================================= softmax warps (both CTAs)
    // Warp w owns the rows of quad w % 4 (TMEM lanes 32 (w % 4) ..) and the
    // KV steps g with g % 2 == w / 4: score buffer, P buffer and every column
    // of the step are its own, so the two warps of a row run a step apart
    // and one's waits overlap the other's arithmetic.  They share one
    // reference maximum per row (shared memory, log2 units), decided in step
    // order: at step g the owner waits for the decision of step g - 1 (the
    // other warp's), lets the reference grow only past the lazy-rescale
    // threshold (then rescales O, after the PV MMA of step g - 1), publishes
    // it, and exponentiates with it.  Each warp keeps its own row sum with
    // the reference it is expressed in; the epilogue combines the two.
    const int quad = warp & 3;
    const int par = warp >> 2;       // steps g with g % 2 == par
    const int r = quad * 32 + lane;  // row of this CTA's tile = TMEM lane
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t t_s = tmem + lane_off + L::t_s + par * 128;  // this warp's score buffer
    const uint32_t t_o = tmem + lane_off + L::t_o;
    const uint32_t t_p = tmem + lane_off + L::t_p + par * 64;   // this warp's P buffer
    float *mref = reinterpret_cast<float *>(smem + L::mref_off);
    float *xsum = reinterpret_cast<float *>(smem + L::xsum_off);
    float *xm = reinterpret_cast<float *>(smem + L::xm_off);
    const float sl2 = p.scale_log2;
    bool ok = true;
    int g = 0, nitem = 0;  // steps and non-empty items so far
    for (int item = cluster; item < p.total_ctas && ok; item += stride) {
      Item it;
      decode(item, it);
      const PairDesc &pd = *it.pd;
      const int n_kv = it.n_kv;
      const int trow = kRowPair ? (int)rank * kRows + r : r;  // row within the item
      const int qrow = it.i0 + trow;                           // row within the pair's chunk
      const int head = it.h0 + (kRowPair ? 0 : (int)rank);
      const bool valid = trow < it.q_rows;
      float m_own = -INFINITY, l_run = 0.f;  // this warp's row sum and its reference
      // The segment of this warp's next step (persistent launches, whose
      // items may span several pairs); one-pair items use pd directly.
      // Masking of item-local step j: it is partly masked when j >= unm_at,
      // and then this row sees the keys before lim_at - 128 j.  An item of
      // grouped pairs moves both to the segment of step j as it goes.
      int64_t lim_at = pd.kv_len;
      int unm_at = it.n_unmasked;
      if constexpr (!kSegs) {
        if (p.causal) {
          const int64_t c = (int64_t)qrow + pd.delta + 1;
          lim_at = c < lim_at ? c : lim_at;
        }
      }
      [[maybe_unused]] int seg_end = 0;
      [[maybe_unused]] const PairDesc *segp = &pd;
      [[maybe_unused]] int seg_left = it.n_segs;
      [[maybe_unused]] auto enter_seg = [&](int base) {
        const Seg q = seg_steps(*segp, it.i0, it.q_rows);
        int64_t lm = segp->kv_len;
        if (p.causal) {
          const int64_t c = (int64_t)qrow + segp->delta + 1;
          lm = c < lm ? c : lm;
        }
        lim_at = lm + (int64_t)base * kKeys;
        unm_at = base + q.n_unmasked;
        seg_end = base + q.n_kv;
      };
      if constexpr (kSegs) enter_seg(0);
      for (int j = (par - g) & 1; j < n_kv; j += 2) {
        if constexpr (kSegs) {
          while (j >= seg_end && seg_left > 1) {
            ++segp;
            --seg_left;
            enter_seg(seg_end);
          }
        }
        const int gj = g + j;
        // Warp-uniform outcome: the TMEM accesses below are warp-collective.
        if (!__all_sync(0xffffffffu, wait(bar(L::b_sfull + par), (gj >> 1) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        float s[kKeys];
        {
          uint32_t sr[kKeys];
          tmem_ld_x128(t_s, sr);
#pragma unroll
          for (int c = 0; c < kKeys; ++c) s[c] = __uint_as_float(sr[c]);
        }
        // The scores are in registers: S(gj + 2) may overwrite the buffer.
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(lead_bar(L::b_sfree + par));
        if (j >= unm_at) {
          const int64_t nv = lim_at - (int64_t)j * kKeys;
          const int nvis = nv < 0 ? 0 : (nv > kKeys ? kKeys : (int)nv);
#pragma unroll
          for (int c = 0; c < kKeys; ++c)
            if (c >= nvis) s[c] = -INFINITY;
        }
        // Row max: eight independent chains of 3-input maxima.
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
        // The reference after step gj - 1 (a new item starts from -inf, but
        // still waits so that the reference is written in step order).
        if (gj > 0 && !__all_sync(0xffffffffu, wait(bar(L::b_dec + quad), (gj - 1) & 1))) {
          ok = false;
          break;
        }
        float m_ref = j == 0 ? -INFINITY : mref[r];
        const float m_new = fmaxf(m_ref, mx * sl2);
        const bool grow = m_new > m_ref + kRescaleLog2;
        const float alpha = grow ? ex2(m_ref - m_new) : 1.f;  // 0 when m_ref = -inf
        const bool rescale_o = grow && m_ref != -INFINITY;   // O holds earlier steps
        if (grow) m_ref = m_new;
        mref[r] = m_ref;
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::b_dec + quad));
        // This warp's row sum follows the reference.
        if (m_own != m_ref) {
          l_run = m_own == -INFINITY ? 0.f : l_run * ex2(m_own - m_ref);
          m_own = m_ref;
        }
        if (__any_sync(0xffffffffu, rescale_o)) {
          // O holds the PV of step gj - 1 only once that MMA is complete (its
          // commit releases K/V stage (gj - 1) % kStages).
          if (!__all_sync(0xffffffffu, wait(bar(L::b_kvempty + (gj - 1) % kStages),
                                            ((gj - 1) / kStages) & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          // Eight columns at a time, not unrolled: the 128 scores stay live
          // across this rarely taken branch.
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
        // p = 2^(s * scale * log2e - m_ref): scale-and-shift two columns per
        // instruction (f32x2 FMA), the row sum in four f32x2 chains; each
        // 32-column quarter of P is stored (16 packed columns) as soon as it
        // exists.
        const float neg_m = m_ref == -INFINITY ? 0.f : -m_ref;
        const float2 sl2v = make_float2(sl2, sl2);
        const float2 negm = make_float2(neg_m, neg_m);
        float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                         make_float2(0.f, 0.f)};
        // P buffer par was last read by PV(gj - 2); its commit released K/V
        // stage (gj - 2) % kStages.
        if (gj >= 2 &&
            !__all_sync(0xffffffffu, wait(bar(L::b_kvempty + (gj - 2) % kStages),
                                          ((gj - 2) / kStages) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int qq = 0; qq < kKeys / 32; ++qq) {
          uint32_t pk[16];
#pragma unroll
          for (int c = qq * 32; c < qq * 32 + 32; c += 2) {
            const float2 x = __ffma2_rn(make_float2(s[c], s[c + 1]), sl2v, negm);
            const float2 pv = make_float2(ex2(x.x), ex2(x.y));
            acc[(c >> 1) & 3] = __fadd2_rn(acc[(c >> 1) & 3], pv);
            pk[(c >> 1) - qq * 16] = pack_bf16(pv.x, pv.y);
          }
          tmem_st_x16(t_p + qq * 16, pk);
        }
        const float2 a01 = __fadd2_rn(acc[0], acc[1]);
        const float2 a23 = __fadd2_rn(acc[2], acc[3]);
        const float2 a03 = __fadd2_rn(a01, a23);
        l_run += a03.x + a03.y;
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(lead_bar(L::b_pready + par));
      }
      if (!ok) break;

      // ---- epilogue: O / l, LSE, routed by the pair's role
      if (n_kv > 0) {
        if (!__all_sync(0xffffffffu, wait(bar(L::b_ofull), nitem & 1))) { ok = false; break; }
        tc_fence_after();
      }
      // One launch for all Pass-KV steps: accumulator updates of a 128-row
      // tile happen in visit order (progress counter per tile, head, batch;
      // each of the tile's softmax warps adds 1 once its part is written).
      int32_t *dep = nullptr;
      if (kPersistent && p.dep_counters != nullptr &&
          (pd.mode == kAccInit || pd.mode == kAccMerge || pd.mode == kAccFinal))
        dep = p.dep_counters + pd.dep_base +
              ((int64_t)(kRowPair ? it.qt * 2 + (int)rank : it.qt) * p.Hq + head) * p.B + it.b;
      if (kDebugChecks && dep != nullptr &&
          (dep < p.dep_counters || dep >= p.dep_counters + p.n_dep_counters)) {
        if (lane == 0) atomicOr(&g_attn_pair_status, kStatusBounds);
        dep = nullptr;
      }
      if (dep != nullptr && pd.visit > 0) {
        int got = 1;
        if (lane == 0) {
          const int target = L::kSoftmaxWarps * pd.visit + p.dep_hold;
          const unsigned long long t0 = global_ns();
          for (uint32_t spin = 0;; ++spin) {
            int v;
            asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(dep) : "memory");
            if (v >= target) break;
            if ((spin & 63u) == 63u && (*abort_flag || global_ns() - t0 > wait_ns)) {
              if (!*abort_flag) {
                *abort_flag = 1;
                asm volatile("st.relaxed.cluster.shared::cluster.u32 [%0], %1;" ::"r"(peer_abort),
                             "r"(1)
                             : "memory");
                atomicOr(&g_attn_pair_status, 1u);
              }
              got = 0;
              break;
            }
          }
        }
        __syncwarp();
        if (!__shfl_sync(0xffffffffu, got, 0)) { ok = false; break; }
      }
      // Both warps of a row read the accumulator's LSE before the exchange
      // below, after which warp par 0 may overwrite it with the merged LSE.
      const float acc_lse_old = valid ? RowSink::acc_lse(p, pd, it.b, head, qrow) : -INFINITY;
      // The row's sum: both warps' sums brought to the final reference (the
      // larger of the two; the reference only grows), added in one order.
      float m_fin = m_own, l_tot = l_run;
      if (n_kv > 0) {
        xsum[par * kRows + r] = l_run;
        xm[par * kRows + r] = m_own;
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::b_xsum + quad));
        if (!__all_sync(0xffffffffu, wait(bar(L::b_xsum + quad), nitem & 1))) { ok = false; break; }
        const float m0 = xm[r], m1 = xm[kRows + r];
        m_fin = fmaxf(m0, m1);
        l_tot = 0.f;
        if (m_fin != -INFINITY) {
          if (m0 != -INFINITY) l_tot += xsum[r] * ex2(m0 - m_fin);
          if (m1 != -INFINITY) l_tot += xsum[kRows + r] * ex2(m1 - m_fin);
        }
      }
      const float inv_l = l_tot > 0.f ? 1.f / l_tot : 0.f;
      const float lse = l_tot > 0.f ? (m_fin + log2f(l_tot)) * 0.6931471805599453f : -INFINITY;
      RowSink sink;
      if (valid) sink.init(p, pd, it.b, head, qrow, lse, par == 0, -1, &acc_lse_old, &g_attn_pair_status);
      // Warp par writes output columns [64 par, 64 par + 64).
#pragma unroll 1
      for (int cc = 0; cc < 2; ++cc) {
        const int c0 = par * 64 + cc * 32;
        float ov[32];
        if (n_kv > 0) {
          uint32_t raw[32];
          tmem_ld_x32(t_o + c0, raw);
#pragma unroll
          for (int x = 0; x < 32; ++x) ov[x] = __uint_as_float(raw[x]) * inv_l;
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x) ov[x] = 0.f;
        }
        if (valid) sink.put<32>(c0, ov);
      }
      if (kPersistent && n_kv > 0) {
        // O has been read: the next item's first PV may overwrite it.
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(lead_bar(L::b_ofree));
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
  cluster_sync();  // neither CTA leaves while the other may still signal it
  if (warp == L::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc_2(tmem, L::kTmemCols);
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

// [b, s, h, 128] bf16 view -> 5-D tensor map (d % 64, s, d / 64, h, b), box
// 64 x box_s x 2 x 1 x 1: one copy brings both 64-column halves of box_s
// rows, half 1 box_s * 128 bytes after half 0, each half in the 128-byte
// swizzled row layout of a separate 64-column copy.
bool make_map_halves(CUtensorMap *map, const void *base, int64_t B, int64_t S, int64_t H,
                     int64_t sb, int64_t ss, int64_t sh, uint32_t box_s) {
  EncodeTiledFn enc = get_encode_fn();
  if (enc == nullptr) return false;
  if (B == 1) sb = S * ss > 0 ? S * ss : 8;  // unused extent: any legal stride
  cuuint64_t dims[5] = {64, (cuuint64_t)S, 2, (cuuint64_t)H, (cuuint64_t)B};
  cuuint64_t strides[4] = {(cuuint64_t)ss * 2, 128, (cuuint64_t)sh * 2, (cuuint64_t)sb * 2};
  cuuint32_t box[5] = {64, box_s, 2, 1, 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// [b, s, h, d] bf16 view -> 4-D tensor map (d, h, s, b), box 64 x 1 x box_s x 1.
bool make_map(CUtensorMap *map, const void *base, int64_t B, int64_t S, int64_t H, int64_t D,
              int64_t sb, int64_t ss, int64_t sh, uint32_t box_s) {
  EncodeTiledFn enc = get_encode_fn();
  if (enc == nullptr) return false;
  if (B == 1) sb = S * ss > 0 ? S * ss : 8;  // unused extent: any legal stride
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)S, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)sh * 2, (cuuint64_t)ss * 2, (cuuint64_t)sb * 2};
  cuuint32_t box[4] = {64, 1, box_s, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <bool kPersistent, bool kRowPair, bool kSegs = false>
cudaError_t launch_pair_t(AttnParams &p, cudaStream_t stream) {
  using L = PairLayout;
  auto kernel = attn_pair_kernel<kPersistent, kRowPair, kSegs>;
  int total = 0;
  if (p.pair_table != nullptr) {
    total = p.total_ctas;  // device-resident table: the caller set cta_begin / n_qtiles
  } else {
    const int rows = kRowPair ? 2 * kRows : kRows, heads = kRowPair ? 1 : 2;
    for (int x = 0; x < p.n_pairs; ++x) {
      PairDesc &pd = p.pairs[x];
      pd.n_qtiles = (pd.q_len + rows - 1) / rows;
      pd.cta_begin = total;
      total += pd.n_qtiles * (p.Hq / heads) * p.B;
    }
    p.total_ctas = total;
  }
  if (total == 0) return cudaSuccess;
  CUtensorMap mq, mk, mv;
  if (!make_map_halves(&mq, p.q, p.B, p.q_rows_total, p.Hq, p.q_sb, p.q_ss, p.q_sh, kRows) ||
      !make_map_halves(&mk, p.k, p.B, p.kv_rows_total, p.Hkv, p.k_sb, p.k_ss, p.k_sh, 64) ||
      !make_map(&mv, p.v, p.B, p.kv_rows_total, p.Hkv, kD, p.v_sb, p.v_ss, p.v_sh, kKeys))
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  int n_attr = 1;
  if (p.dep_counters != nullptr) {
    // CTAs wait on other CTAs' progress counters: they must all be resident.
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = 1;
    n_attr = 2;
  }
  cfg.blockDim = dim3(L::kThreads);
  cfg.dynamicSmemBytes = L::alloc_bytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = n_attr;
  // Per device, once: the kernel's shared-memory attribute and how many CTA
  // pairs fit on the GPU at once (the grid of a persistent launch).
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static bool configured[kMaxDevices] = {};
  static int max_clusters[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return cudaErrorInvalidDevice;
  int fit = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!configured[dev]) {
      cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           L::alloc_bytes);
      if (e != cudaSuccess) return e;
      cudaLaunchConfig_t occ = cfg;
      occ.gridDim = dim3(2);
      occ.numAttrs = 1;  // cluster shape only
      e = cudaOccupancyMaxActiveClusters(&max_clusters[dev], kernel, &occ);
      if (e != cudaSuccess) return e;
      configured[dev] = true;
    }
    fit = max_clusters[dev];
  }
  int clusters = total;
  if (kPersistent) {
    if (fit < 1) return cudaErrorInvalidConfiguration;
    clusters = fit < total ? fit : total;
    p.persistent_ctas = clusters;
  }
  cfg.gridDim = dim3(2 * clusters);
  return cudaLaunchKernelEx(&cfg, kernel, mq, mk, mv, p);
}

cudaError_t launch_pair_any(AttnParams &p, cudaStream_t stream) {
  const bool pers = p.persistent_ctas > 0;
  if (p.seg_groups) {
    // Grouped pairs (on-chip accumulation across a query piece's K/V pieces):
    // persistent launches only, in their own kernel instance.
    if (!pers || p.pair_table == nullptr) return cudaErrorInvalidValue;
    return p.row_pair ? launch_pair_t<true, true, true>(p, stream)
                      : launch_pair_t<true, false, true>(p, stream);
  }
  if (p.row_pair)
    return pers ? launch_pair_t<true, true>(p, stream) : launch_pair_t<false, true>(p, stream);
  return pers ? launch_pair_t<true, false>(p, stream) : launch_pair_t<false, false>(p, stream);
}

}  // namespace

cudaError_t launch_attn_pair(AttnParams &p, cudaStream_t stream) {
  p.row_pair = (p.Hq / p.Hkv) % 2 != 0 ? 1 : 0;
  return launch_pair_any(p, stream);
}

bool attn_tc_supported(const AttnParams &p) {
  if (p.pack_g > 0) return attn_decode_tc_supported(p);
  return !p.in_f32 && p.D == kD && p.q_rows_total > 0 && p.kv_rows_total > 0;
}

TcItemShape attn_tc_item_shape(const AttnParams &p) {
  if (p.pack_g > 0) return {kRows, 1};
  return (p.Hq / p.Hkv) % 2 == 0 ? TcItemShape{kRows, 2} : TcItemShape{2 * kRows, 1};
}

cudaError_t launch_attn_tc(AttnParams &p, cudaStream_t stream) {
  return p.pack_g > 0 ? launch_attn_decode_tc(p, stream) : launch_attn_pair(p, stream);
}

unsigned int attn_pair_read_status(bool clear, cudaError_t *err) {
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_attn_pair_status, sizeof(v));
  if (e == cudaSuccess && clear) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_attn_pair_status, &zero, sizeof(zero));
  }
  if (err) *err = e;
  return v;
}

}  // namespace cpattn
