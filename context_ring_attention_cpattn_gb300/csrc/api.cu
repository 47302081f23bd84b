// C ABI of libcpattn.so: argument checks, the CP ring plan, workspace layout
// and the step-by-step launch sequence (see include/cpattn.h).
//
// The ring emulation follows "Scaling LLM Inference ..." (techreport rewrite,
// section "Context Parallelism for Million-Token Contexts"): the sequence is
// split into N chunks, one per CP rank.  Pass-KV keeps Q chunk r on rank r
// and moves K/V chunks around the ring: at step t rank r holds K/V chunk
// (r - t) mod N and folds its pair into a running (O, LSE) accumulator.
// Pass-Q keeps K/V chunk r on rank r and moves the Q chunks: at step t rank r
// sees Q chunk (r - t) mod N and stores that pair's partial; after the ring
// every Q chunk's partials are merged by LSE.  On one GPU a "rank" is a pair
// in a launch, a "send" is a different row offset into the resident tensors,
// and the N ring steps are N launches back to back on one stream.
#include <cuda_runtime.h>
#include <math.h>
#include <nvtx3/nvToolsExt.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <functional>
#include <new>
#include <vector>

#include "cpattn_internal.h"

using namespace cpattn;

namespace {

// ----------------------------------------------------------------- checks
int elem_bytes(int32_t dtype) {
  return dtype == CPATTN_BF16 ? 2 : (dtype == CPATTN_FP32 ? 4 : 0);
}

constexpr int64_t kMaxRows = (int64_t)1 << 30;

// Shape, dtype, pointer and stride checks shared by every tensor argument.
cpattn_status check_view(const cpattn_tensor *t) {
  if (t == nullptr) return CPATTN_ERR_INVALID_ARG;
  const int es = elem_bytes(t->dtype);
  if (es == 0) return CPATTN_ERR_INVALID_ARG;
  if (t->b < 1 || t->s < 0 || t->h < 1 || t->d < 1) return CPATTN_ERR_INVALID_ARG;
  if (t->s > kMaxRows || t->b > 65535 || t->h > 65535) return CPATTN_ERR_UNSUPPORTED;
  if (t->s > 0 && t->data == nullptr) return CPATTN_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(t->data) % 16 != 0) return CPATTN_ERR_INVALID_ARG;
  if (t->stride_h < 0 || t->stride_s < 0 || t->stride_b < 0) return CPATTN_ERR_INVALID_ARG;
  if ((t->stride_h * es) % 16 != 0 || (t->stride_s * es) % 16 != 0) return CPATTN_ERR_INVALID_ARG;
  if (t->b > 1 && (t->stride_b * es) % 16 != 0) return CPATTN_ERR_INVALID_ARG;
  if (t->h > 1 && t->stride_h < t->d) return CPATTN_ERR_INVALID_ARG;
  return CPATTN_OK;
}

// q, k, v consistency.
cpattn_status check_qkv(const cpattn_tensor *q, const cpattn_tensor *k, const cpattn_tensor *v) {
  cpattn_status s;
  if ((s = check_view(q)) != CPATTN_OK) return s;
  if ((s = check_view(k)) != CPATTN_OK) return s;
  if ((s = check_view(v)) != CPATTN_OK) return s;
  if (k->dtype != q->dtype || v->dtype != q->dtype) return CPATTN_ERR_INVALID_ARG;
  if (k->b != q->b || v->b != q->b) return CPATTN_ERR_INVALID_ARG;
  if (v->s != k->s || v->h != k->h) return CPATTN_ERR_INVALID_ARG;
  if (k->d != q->d || v->d != q->d) return CPATTN_ERR_INVALID_ARG;
  if (q->h % k->h != 0) return CPATTN_ERR_INVALID_ARG;
  if (q->d != 64 && q->d != 128) return CPATTN_ERR_UNSUPPORTED;
  return CPATTN_OK;
}

cpattn_status check_out(const cpattn_tensor *o, const float *lse, const cpattn_tensor *q) {
  cpattn_status s = check_view(o);
  if (s != CPATTN_OK) return s;
  if (o->b != q->b || o->s != q->s || o->h != q->h || o->d != q->d) return CPATTN_ERR_INVALID_ARG;
  if (q->s > 0 && lse == nullptr) return CPATTN_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(lse) % 4 != 0) return CPATTN_ERR_INVALID_ARG;
  return CPATTN_OK;
}

float resolve_scale(float scale, int64_t d) {
  return scale > 0.f ? scale : (float)(1.0 / sqrt((double)d));
}

OutView out_view(const cpattn_tensor *o, float *lse) {
  OutView w;
  memset(&w, 0, sizeof(w));
  w.o = o->data;
  w.lse = lse;
  w.sb = o->stride_b;
  w.ss = o->stride_s;
  w.sh = o->stride_h;
  w.lb = o->h * o->s;
  w.lh = o->s;
  w.f32 = o->dtype == CPATTN_FP32;
  return w;
}

void fill_inputs(AttnParams &p, const cpattn_tensor *q, const cpattn_tensor *k,
                 const cpattn_tensor *v, int causal, float scale) {
  memset(&p, 0, sizeof(p));
  p.B = (int32_t)q->b;
  p.Hq = (int32_t)q->h;
  p.Hkv = (int32_t)k->h;
  p.D = (int32_t)q->d;
  p.causal = causal ? 1 : 0;
  p.scale = resolve_scale(scale, q->d);
  p.scale_log2 = (float)((double)p.scale * 1.4426950408889634);
  p.q = q->data;
  p.k = k->data;
  p.v = v->data;
  p.q_sb = q->stride_b; p.q_ss = q->stride_s; p.q_sh = q->stride_h;
  p.k_sb = k->stride_b; p.k_ss = k->stride_s; p.k_sh = k->stride_h;
  p.v_sb = v->stride_b; p.v_ss = v->stride_s; p.v_sh = v->stride_h;
  p.q_rows_total = q->s;
  p.kv_rows_total = k->s;
  p.in_f32 = q->dtype == CPATTN_FP32;
}

// Number of (query, key) pairs the mask keeps for query rows at positions
// q0 .. q0+nq-1 against keys at k0 .. k0+nk-1.
double visible_pairs(int64_t q0, int64_t nq, int64_t k0, int64_t nk, bool causal) {
  if (nq <= 0 || nk <= 0) return 0.0;
  if (!causal) return (double)nq * (double)nk;
  const int64_t a = q0 - k0 + 1;  // keys visible to row i: clamp(a + i, 0, nk)
  const int64_t lo = std::min<int64_t>(std::max<int64_t>(1 - a, 0), nq);
  const int64_t hi = std::min<int64_t>(std::max<int64_t>(nk - a, lo), nq);
  const double ramp = (double)(hi - lo) * (double)a + (double)(lo + hi - 1) * (double)(hi - lo) / 2.0;
  return ramp + (double)(nq - hi) * (double)nk;
}

// ----------------------------------------------------------------- tracing
// An NVTX range around the enqueue of each ring step, merge and entry point
// ("cpattn pass_kv step 3", "cpattn pass_q merge", ...): profilers attribute
// the kernels launched inside a range to it, which ties a launch list to the
// ring's steps.  Without a tool attached a range costs a few nanoseconds.
struct NvtxRange {
  explicit NvtxRange(const char *fmt, ...) {
    char buf[96];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    nvtxRangePushA(buf);
  }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange &) = delete;
  NvtxRange &operator=(const NvtxRange &) = delete;
};

const char *mode_name(int mode) { return mode == CPATTN_PASS_Q ? "pass_q" : "pass_kv"; }

// ----------------------------------------------------------------- profiling
struct Profiler {
  bool armed = false;
  int capacity = 0;
  int n = 0;
  std::vector<cudaEvent_t> events;
  std::vector<int32_t> kinds;
  std::vector<double> work;
};
Profiler g_prof;

void prof_before(cudaStream_t st) {
  if (g_prof.armed && g_prof.n < g_prof.capacity) cudaEventRecord(g_prof.events[2 * g_prof.n], st);
}
void prof_after(cudaStream_t st, int kind, double work) {
  if (g_prof.armed && g_prof.n < g_prof.capacity) {
    cudaEventRecord(g_prof.events[2 * g_prof.n + 1], st);
    g_prof.kinds[g_prof.n] = kind;
    g_prof.work[g_prof.n] = work;
    ++g_prof.n;
  }
}

// ----------------------------------------------------------------- plan table upload
// The single-launch mode reads its pair table from the workspace.  The table
// travels in the parameter blocks of small fill kernels (kTableChunk entries
// each), which the driver copies at launch: no host buffer has to outlive the
// call, nothing waits on the host, and the upload can be captured in a graph.
constexpr int kTableChunk = 80;
struct TableChunk {
  PairDesc *dst;
  int32_t n;
  int32_t pad;
  PairDesc e[kTableChunk];
};
static_assert(sizeof(TableChunk) <= 4096, "fill kernel parameters too large");

__global__ void table_fill_kernel(const __grid_constant__ TableChunk c) {
  const int i = (int)threadIdx.x;
  if (i < c.n) c.dst[i] = c.e[i];
}

cudaError_t upload_table(PairDesc *dst, const std::vector<PairDesc> &table, cudaStream_t st) {
  for (size_t x0 = 0; x0 < table.size(); x0 += kTableChunk) {
    TableChunk c;
    memset(&c, 0, sizeof(c));
    c.dst = dst + x0;
    c.n = (int32_t)std::min<size_t>(kTableChunk, table.size() - x0);
    for (int i = 0; i < c.n; ++i) c.e[i] = table[x0 + i];
    prof_before(st);
    table_fill_kernel<<<1, 128, 0, st>>>(c);
    prof_after(st, CPATTN_KERNEL_TABLE, (double)c.n * sizeof(PairDesc));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// ----------------------------------------------------------------- the plan
// The sequence is cut into pieces; rank r of N holds piece r (contiguous
// assignment) or pieces r and 2N-1-r (zigzag assignment, which gives every
// rank the same causal work).  Q and K/V use the same assignment.
struct Plan {
  int N = 0;
  int mode = 0;
  int assign = CPATTN_ASSIGN_CONTIGUOUS;
  int P = 0;                               // pieces per sequence
  int64_t Cq = 0, C = 0;                   // Q and K/V piece lengths
  std::vector<cpattn_plan_entry> entries;  // launch order
  int n_launches = 0;
  std::vector<int> count;                  // visible K/V pieces per Q piece
  std::vector<int> slot0;                  // Pass-Q: first slot of the Q piece (-1: none)
  int n_slots = 0;
  bool need_acc = false;                   // Pass-KV needs the accumulator
};

int rank_pieces(const Plan &pl, int r, int out[2]) {
  if (pl.assign == CPATTN_ASSIGN_ZIGZAG) {
    out[0] = r;
    out[1] = 2 * pl.N - 1 - r;
    return 2;
  }
  out[0] = r;
  return 1;
}

bool pair_visible(const Plan &pl, int64_t q_base, bool causal, int i, int j) {
  if (pl.Cq <= 0 || pl.C <= 0) return false;
  if (!causal) return true;
  return (int64_t)j * pl.C <= q_base + (int64_t)i * pl.Cq + pl.Cq - 1;
}

cpattn_status build_plan(int64_t sq, int64_t skv, int64_t q_base, int n_chunks, int mode,
                         int causal, int assign, Plan &pl) {
  if (n_chunks < 1 || n_chunks > kMaxPairs) return CPATTN_ERR_INVALID_ARG;
  if (mode != CPATTN_PASS_KV && mode != CPATTN_PASS_Q) return CPATTN_ERR_INVALID_ARG;
  if (assign != CPATTN_ASSIGN_CONTIGUOUS && assign != CPATTN_ASSIGN_ZIGZAG)
    return CPATTN_ERR_INVALID_ARG;
  const int P = assign == CPATTN_ASSIGN_ZIGZAG ? 2 * n_chunks : n_chunks;
  if (sq < 0 || skv < 0 || sq % P != 0 || skv % P != 0) return CPATTN_ERR_INVALID_ARG;
  if (sq > kMaxRows || skv > kMaxRows || q_base < -kMaxRows * 4 || q_base > kMaxRows * 4)
    return CPATTN_ERR_UNSUPPORTED;
  // Pairs per launch: N (contiguous), 2N (zigzag Pass-KV), 4N (zigzag Pass-Q).
  const int per_launch = assign == CPATTN_ASSIGN_ZIGZAG ? (mode == CPATTN_PASS_Q ? 4 : 2) : 1;
  if (per_launch * n_chunks > kMaxPairs) return CPATTN_ERR_UNSUPPORTED;
  const int N = n_chunks;
  pl.N = N;
  pl.mode = mode;
  pl.assign = assign;
  pl.P = P;
  pl.Cq = sq / P;
  pl.C = skv / P;
  pl.count.assign(P, 0);
  pl.slot0.assign(P, -1);
  pl.entries.clear();
  for (int i = 0; i < P; ++i)
    for (int j = 0; j < P; ++j) pl.count[i] += pair_visible(pl, q_base, causal, i, j) ? 1 : 0;
  pl.n_slots = 0;
  if (mode == CPATTN_PASS_Q) {
    for (int i = 0; i < P; ++i)
      if (pl.count[i] >= 2) {
        pl.slot0[i] = pl.n_slots;
        pl.n_slots += pl.count[i];
      }
  }
  std::vector<int> seen(P, 0);
  int launch = 0;
  auto emit = [&](int t, int r, int i, int j) {
    if (!pair_visible(pl, q_base, causal, i, j)) return;
    cpattn_plan_entry e;
    e.step = t;
    e.q_chunk = i;
    e.kv_chunk = j;
    e.slot = -1;
    e.launch = launch;
    e.rank = r;
    if (pl.count[i] == 1) {
      e.role = CPATTN_ROLE_STORE;
    } else if (mode == CPATTN_PASS_KV) {
      const int k = seen[i]++;
      e.role = k == 0 ? CPATTN_ROLE_ACC_INIT
                      : (k == pl.count[i] - 1 ? CPATTN_ROLE_ACC_FINAL : CPATTN_ROLE_ACC_MERGE);
      pl.need_acc = true;
    } else {
      int rank = 0;  // position of j among piece i's visible K/V pieces, ascending
      for (int jj = 0; jj < j; ++jj) rank += pair_visible(pl, q_base, causal, i, jj) ? 1 : 0;
      e.role = CPATTN_ROLE_PARTIAL;
      e.slot = pl.slot0[i] + rank;
    }
    pl.entries.push_back(e);
  };
  for (int t = 0; t < N; ++t) {
    if (mode == CPATTN_PASS_KV) {
      // Rank r keeps its Q pieces and receives the K/V pieces of rank
      // (r - t) mod N.  Each K/V piece of the visiting rank is its own launch,
      // so no Q piece's accumulator is updated twice in one launch.
      const int n_sub = assign == CPATTN_ASSIGN_ZIGZAG ? 2 : 1;
      for (int u = 0; u < n_sub; ++u) {
        const size_t before = pl.entries.size();
        for (int r = 0; r < N; ++r) {
          int qp[2], kp[2];
          const int nq = rank_pieces(pl, r, qp);
          rank_pieces(pl, ((r - t) % N + N) % N, kp);
          for (int a = 0; a < nq; ++a) emit(t, r, qp[a], kp[u]);
        }
        if (pl.entries.size() > before) ++launch;
      }
    } else {
      // Rank r keeps its K/V pieces and receives the Q pieces of rank (r - t) mod N.
      const size_t before = pl.entries.size();
      for (int r = 0; r < N; ++r) {
        int qp[2], kp[2];
        const int nq = rank_pieces(pl, ((r - t) % N + N) % N, qp);
        const int nk = rank_pieces(pl, r, kp);
        for (int a = 0; a < nq; ++a)
          for (int b = 0; b < nk; ++b) emit(t, r, qp[a], kp[b]);
      }
      if (pl.entries.size() > before) ++launch;
    }
  }
  pl.n_launches = launch;
  return CPATTN_OK;
}

// Work of every (ring step, rank) in visible (query, key) pairs per head:
// a real ring step lasts as long as its busiest rank.
void plan_work(const Plan &pl, int64_t q_base, bool causal, std::vector<double> &step_max,
               double &critical, double &total) {
  std::vector<double> w((size_t)pl.N * pl.N, 0.0);
  total = 0.0;
  for (const auto &e : pl.entries) {
    const double v = visible_pairs(q_base + (int64_t)e.q_chunk * pl.Cq, pl.Cq,
                                   (int64_t)e.kv_chunk * pl.C, pl.C, causal);
    w[(size_t)e.step * pl.N + e.rank] += v;
    total += v;
  }
  step_max.assign(pl.N, 0.0);
  critical = 0.0;
  for (int t = 0; t < pl.N; ++t) {
    for (int r = 0; r < pl.N; ++r) step_max[t] = std::max(step_max[t], w[(size_t)t * pl.N + r]);
    critical += step_max[t];
  }
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsLayout {
  size_t acc_o = 0, acc_lse = 0;      // Pass-KV
  size_t part_o = 0, part_lse = 0;    // Pass-Q
  int64_t slot_o_elems = 0, slot_lse_elems = 0;
  size_t table = 0, counters = 0;     // one launch for all steps
  size_t n_counters = 0;
  size_t total = 0;
};

// 128-row query tiles of a Q piece, rounded up to whole 256-row pairs (the
// row-pair work items of odd GQA groups index their tiles up to there).
int64_t tiles_per_piece(const Plan &pl) { return 2 * ((pl.Cq + 255) / 256); }

WsLayout ws_layout(const Plan &pl, int64_t B, int64_t sq, int64_t hq, int64_t d,
                   int launch_mode = CPATTN_LAUNCH_PER_STEP) {
  WsLayout w;
  size_t off = 0;
  const bool onchip = launch_mode == CPATTN_LAUNCH_SINGLE_ONCHIP && pl.mode == CPATTN_PASS_KV;
  if (launch_mode == CPATTN_LAUNCH_SINGLE || launch_mode == CPATTN_LAUNCH_SINGLE_ONCHIP) {
    w.table = off;
    off = align256(off + pl.entries.size() * sizeof(PairDesc));
  }
  if (launch_mode == CPATTN_LAUNCH_SINGLE) {
    w.counters = off;
    w.n_counters = (size_t)pl.P * tiles_per_piece(pl) * hq * B;
    off = align256(off + w.n_counters * sizeof(int32_t));
  }
  if (pl.mode == CPATTN_PASS_KV && pl.need_acc && !onchip) {
    w.acc_o = off;
    off = align256(off + (size_t)B * sq * hq * d * 4);
    w.acc_lse = off;
    off = align256(off + (size_t)B * hq * sq * 4);
  }
  if (pl.mode == CPATTN_PASS_Q && pl.n_slots > 0) {
    w.slot_o_elems = B * pl.Cq * hq * d;
    w.slot_lse_elems = B * hq * pl.Cq;
    w.part_o = off;
    off = align256(off + (size_t)pl.n_slots * w.slot_o_elems * 4);
    w.part_lse = off;
    off = align256(off + (size_t)pl.n_slots * w.slot_lse_elems * 4);
  }
  w.total = off;
  return w;
}

cudaError_t launch_attn(AttnParams &p, cudaStream_t st, const cpattn_tensor *q,
                        double vis_override = -1.0) {
  double vis = 0.0;
  for (int x = 0; x < p.n_pairs; ++x) {
    const PairDesc &pd = p.pairs[x];
    vis += visible_pairs(pd.delta, pd.q_len, 0, pd.kv_len, p.causal != 0);
  }
  if (vis_override >= 0.0) vis = vis_override;
  const double flops = 4.0 * (double)q->d * (double)q->h * (double)q->b * vis;
  // Kernel-side waits give up after 2 s, or after four times the launch's
  // whole work at 100 TFLOP/s when that is longer (a wait in a persistent
  // launch can last as long as other CTAs' items).
  p.wait_ns = (uint64_t)std::max(2e9, 4.0 * flops / 1e14 * 1e9);
  const bool tc = attn_tc_supported(p);
  prof_before(st);
  cudaError_t e = tc ? launch_attn_tc(p, st) : launch_attn_simt(p, st);
  prof_after(st,
             !tc ? CPATTN_KERNEL_ATTN_SIMT
                 : (p.seg_groups ? CPATTN_KERNEL_ATTN_TC_ONCHIP : CPATTN_KERNEL_ATTN_TC),
             flops);
  return e;
}

int assignment_of(const cpattn_prefill_options *opts) {
  return opts ? opts->assignment : CPATTN_ASSIGN_CONTIGUOUS;
}

int launch_mode_of(const cpattn_prefill_options *opts) {
  return opts ? opts->launch : CPATTN_LAUNCH_DEFAULT;
}

bool valid_launch(int l) {
  return l == CPATTN_LAUNCH_PER_STEP || l == CPATTN_LAUNCH_PERSISTENT_STEP ||
         l == CPATTN_LAUNCH_SINGLE || l == CPATTN_LAUNCH_AUTO || l == CPATTN_LAUNCH_SINGLE_ONCHIP;
}

// CPATTN_LAUNCH_AUTO: one persistent launch for all ring steps when work
// items are short (mean visible 128-key tiles per 128-row query tile below
// kAutoSingleTiles), where each CTA's start-up and write-out is a large share
// of its work; one launch per step otherwise.  Measured on GB300 (TFLOP/s,
// per step vs single): 8-tile items 589 vs 687, 32-tile 922 vs 1036,
// 60-tile 1367 vs 1304.
constexpr double kAutoSingleTiles = 48.0;
// K/V bytes up to which an on-chip Pass-KV launch keeps its K/V reads in L2
// (the GPU has 126 MB).
constexpr double kOnchipKvBytes = 96.0 * 1024 * 1024;

// Work items are short when a 128-row query tile sees, on average over the
// ring's pairs, fewer than kAutoSingleTiles visible 128-key tiles.
bool short_items(const Plan &pl, int64_t q_base, int causal) {
  double vis = 0.0, rows = 0.0;
  for (const auto &e : pl.entries) {
    const int64_t delta = q_base + (int64_t)e.q_chunk * pl.Cq - (int64_t)e.kv_chunk * pl.C;
    vis += visible_pairs(delta, pl.Cq, 0, pl.C, causal != 0);
    rows += (double)pl.Cq;
  }
  const double tiles = rows > 0.0 ? vis / rows / 128.0 : 0.0;
  return tiles < kAutoSingleTiles;
}

int resolve_launch(int lmode, const Plan &pl, const cpattn_tensor *q, const cpattn_tensor *k,
                   int64_t q_base, int causal) {
  if (lmode != CPATTN_LAUNCH_AUTO) return lmode;
  if (q->dtype != CPATTN_BF16 || q->d != 128) return CPATTN_LAUNCH_PER_STEP;  // no tensor-core kernel
  const bool short_it = short_items(pl, q_base, causal);
  if (pl.mode == CPATTN_PASS_KV) {
    // The accumulator on chip (no fp32 round trip per visit) when items are
    // short or K and V stay in L2: an on-chip item streams its own sequence
    // of K/V pieces, so concurrent items read different pieces, which L2 can
    // hold only for a small K/V.  Measured on one GB300: 128K (K/V 64 MiB)
    // 44.5 vs 49.6 ms per layer per step; 1M (K/V 512 MiB) 1718 vs 1362 ms.
    const double kv_bytes = (double)k->b * (double)k->s * (double)k->h * (double)k->d * 2.0 * 2.0;
    return (short_it || kv_bytes <= kOnchipKvBytes) ? CPATTN_LAUNCH_SINGLE_ONCHIP
                                                     : CPATTN_LAUNCH_PER_STEP;
  }
  return short_it ? CPATTN_LAUNCH_SINGLE : CPATTN_LAUNCH_PER_STEP;
}

// Groups of Q pieces for a host-buffer call that streams Q in piece by piece
// and copies output back as it becomes final (long items only; otherwise one
// group of all pieces).  In arrival order: a small first group, so work starts
// once K/V and a few pieces are in; up to three middle groups of about equal
// size, each started once its pieces are in, whose output goes back while the
// later groups run; and the last piece alone, so that only its own output
// (and, for Pass-Q, its merge) is left when the work ends.  A piece's work
// items are the same in every grouping (bitwise-equal results).
std::vector<std::vector<int>> piece_groups(int P, bool split) {
  std::vector<std::vector<int>> groups;
  auto add = [&](int a, int b) {
    groups.emplace_back();
    for (int i = a; i < b; ++i) groups.back().push_back(i);
  };
  if (!split || P < 4) {
    add(0, P);
    return groups;
  }
  const int first = std::max(1, P / 8);
  add(0, first);
  const int middle = P - first - 1, m = std::min(3, middle);
  int at = first;
  for (int x = 0; x < m; ++x) {
    const int size = middle / m + (x >= m - middle % m ? 1 : 0);
    add(at, at + size);
    at += size;
  }
  add(P - 1, P);
  return groups;
}

// Called (at enqueue time, on the host) once the work that finalises output
// rows [row0, row0 + rows) has been enqueued on the stream.
using FinalRowsFn = std::function<cudaError_t(int64_t row0, int64_t rows)>;
// Called before a launch that reads Q piece q_piece and K/V piece kv_piece.
using InputsFn = std::function<cudaError_t(int q_piece, int kv_piece)>;

cpattn_status prefill_impl(const cpattn_tensor *q, const cpattn_tensor *k, const cpattn_tensor *v,
                           int64_t q_base, int n_chunks, int mode, int causal, float scale,
                           cpattn_tensor *o, float *lse, void *workspace, size_t ws_bytes,
                           const cpattn_prefill_options *opts, cudaStream_t st,
                           const FinalRowsFn *on_final = nullptr,
                           const InputsFn *on_inputs = nullptr) {
  cpattn_status s = check_qkv(q, k, v);
  if (s != CPATTN_OK) return s;
  if ((s = check_out(o, lse, q)) != CPATTN_OK) return s;
  Plan pl;
  if ((s = build_plan(q->s, k->s, q_base, n_chunks, mode, causal, assignment_of(opts), pl)) !=
      CPATTN_OK)
    return s;
  int lmode = launch_mode_of(opts);
  if (!valid_launch(lmode)) return CPATTN_ERR_INVALID_ARG;
  lmode = resolve_launch(lmode, pl, q, k, q_base, causal);
  const bool onchip = lmode == CPATTN_LAUNCH_SINGLE_ONCHIP && pl.mode == CPATTN_PASS_KV;
  const bool single = lmode == CPATTN_LAUNCH_SINGLE || lmode == CPATTN_LAUNCH_SINGLE_ONCHIP;
  const WsLayout wl = ws_layout(pl, q->b, q->s, q->h, q->d, lmode);
  if (wl.total > 0) {
    if (workspace == nullptr || ws_bytes < wl.total) return CPATTN_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return CPATTN_ERR_WORKSPACE;
  }
  if (q->s == 0) return CPATTN_OK;
  uint8_t *ws = reinterpret_cast<uint8_t *>(workspace);

  AttnParams p;
  fill_inputs(p, q, k, v, causal, scale);
  p.out = out_view(o, lse);
  if (pl.mode == CPATTN_PASS_KV && pl.need_acc && !onchip) {
    p.acc.o = ws + wl.acc_o;
    p.acc.lse = reinterpret_cast<float *>(ws + wl.acc_lse);
    p.acc.sh = q->d;
    p.acc.ss = q->h * q->d;
    p.acc.sb = q->s * q->h * q->d;
    p.acc.lh = q->s;
    p.acc.lb = q->h * q->s;
    p.acc.f32 = 1;
  }
  p.n_part_slots = pl.n_slots;
  p.part_rows = (int32_t)pl.Cq;
  p.n_dep_counters = (int32_t)wl.n_counters;
  if (pl.n_slots > 0) {
    p.part.o = ws + wl.part_o;
    p.part.lse = reinterpret_cast<float *>(ws + wl.part_lse);
    p.part.sh = q->d;
    p.part.ss = q->h * q->d;
    p.part.sb = pl.Cq * q->h * q->d;
    p.part.lh = pl.Cq;
    p.part.lb = q->h * pl.Cq;
    p.part.f32 = 1;
    p.part_o_stride = wl.slot_o_elems;
    p.part_lse_stride = wl.slot_lse_elems;
  }

  // Pairs of the plan entries `idx` ordered by work, largest first.
  auto launch_items_of = [&](const std::vector<size_t> &idx, std::vector<PairDesc> &out) {
    struct Item { PairDesc pd; double work; };
    std::vector<Item> items;
    for (size_t x : idx) {
      const cpattn_plan_entry &e = pl.entries[x];
      Item it;
      memset(&it.pd, 0, sizeof(it.pd));
      it.pd.q_row0 = (int32_t)(e.q_chunk * pl.Cq);
      it.pd.q_len = (int32_t)pl.Cq;
      it.pd.kv_row0 = (int32_t)(e.kv_chunk * pl.C);
      it.pd.kv_len = (int32_t)pl.C;
      it.pd.delta = q_base + (int64_t)e.q_chunk * pl.Cq - (int64_t)e.kv_chunk * pl.C;
      it.pd.mode = e.role;
      it.pd.slot = e.slot;
      it.pd.dep_base = (int32_t)((int64_t)e.q_chunk * tiles_per_piece(pl) * q->h * q->b);
      it.work = visible_pairs(it.pd.delta, pl.Cq, 0, pl.C, causal != 0);
      items.push_back(it);
    }
    std::stable_sort(items.begin(), items.end(),
                     [](const Item &a, const Item &b) { return a.work > b.work; });
    for (const auto &it : items) out.push_back(it.pd);
  };
  // ... of one launch of the plan: entries [e0, e1).
  auto launch_items = [&](size_t e0, size_t e1, std::vector<PairDesc> &out) {
    std::vector<size_t> idx;
    for (size_t x = e0; x < e1; ++x) idx.push_back(x);
    launch_items_of(idx, out);
  };

  // Host-buffer calls with long items split the on-chip launch into groups
  // of Q pieces (piece_groups); every group's rows go back after its launch.
  const bool grouped = onchip && on_inputs != nullptr && !short_items(pl, q_base, causal);
  if (single && attn_tc_supported(p)) {
    NvtxRange range("cpattn %s ring, one launch%s", mode_name(mode), grouped ? " per group" : "");
    std::vector<PairDesc> table;
    size_t e0 = 0;
    for (int l = 0; l < pl.n_launches; ++l) {
      size_t e1 = e0;
      while (e1 < pl.entries.size() && pl.entries[e1].launch == l) ++e1;
      launch_items(e0, e1, table);
      e0 = e1;
    }
    const TcItemShape sh = attn_tc_item_shape(p);
    const int per_tile = (int)(q->h / sh.heads) * (int)q->b;
    PairDesc *dev_table = reinterpret_cast<PairDesc *>(ws + wl.table);
    // One launch over `lt` (total work items, visible pairs) after its
    // inputs are in; the table goes to dev_table + t_off.
    size_t t_off = 0;
    auto launch_table = [&](const std::vector<PairDesc> &lt, int total, double vis) -> cpattn_status {
      if (total == 0) return CPATTN_OK;
      if (upload_table(dev_table + t_off, lt, st) != cudaSuccess) return CPATTN_ERR_CUDA;
      p.pair_table = dev_table + t_off;
      p.n_table = (int32_t)lt.size();
      p.total_ctas = total;
      p.persistent_ctas = 1;
      p.seg_groups = onchip ? 1 : 0;
      if (pl.mode == CPATTN_PASS_KV && pl.need_acc && !onchip) {
        p.dep_counters = reinterpret_cast<int32_t *>(ws + wl.counters);
        p.dep_hold = (opts != nullptr && opts->hold_ordered_waits != 0) ? (1 << 28) : 0;
        if (cudaMemsetAsync(p.dep_counters, 0, wl.n_counters * sizeof(int32_t), st) != cudaSuccess)
          return CPATTN_ERR_CUDA;
      }
      if (launch_attn(p, st, q, vis) != cudaSuccess) return CPATTN_ERR_CUDA;
      t_off += lt.size();
      p.pair_table = nullptr;
      p.n_table = 0;
      p.dep_counters = nullptr;
      p.dep_hold = 0;
      p.persistent_ctas = 0;
      p.seg_groups = 0;
      return CPATTN_OK;
    };
    if (onchip) {
      // Each Q piece's pairs in ring order form one run of work items: a
      // work item streams every visiting K/V piece through one on-chip
      // accumulator and stores the result (segment x: visit = x, slot = the
      // run's length).  Within a launch, runs with the most work first.
      std::vector<std::vector<PairDesc>> runs(pl.P);
      std::vector<double> work(pl.P, 0.0);
      for (const auto &pd : table) {
        const int piece = (int)(pd.q_row0 / pl.Cq);
        runs[piece].push_back(pd);
        work[piece] += visible_pairs(pd.delta, pd.q_len, 0, pd.kv_len, causal != 0);
      }
      for (const auto &grp : piece_groups(pl.P, grouped)) {
        std::vector<int> order;
        for (int i : grp)
          if (!runs[i].empty()) order.push_back(i);
        std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return work[a] > work[b]; });
        std::vector<PairDesc> lt;
        int total = 0;
        double vis = 0.0;
        for (int i : order) {
          const int n = (int)runs[i].size();
          const int n_qtiles = (runs[i][0].q_len + sh.rows - 1) / sh.rows;
          for (int x = 0; x < n; ++x) {
            PairDesc pd = runs[i][x];
            pd.mode = kStore;
            pd.visit = x;
            pd.slot = n;
            pd.n_qtiles = n_qtiles;
            pd.cta_begin = total;
            lt.push_back(pd);
          }
          total += n_qtiles * per_tile;
          vis += work[i];
        }
        // Inputs arriving piece by piece: the launch reads all of its pieces.
        for (int i : grp)
          if (on_inputs != nullptr && (*on_inputs)(i, 0) != cudaSuccess) return CPATTN_ERR_CUDA;
        if ((s = launch_table(lt, total, vis)) != CPATTN_OK) return s;
        for (int i : order)
          if (grouped && on_final != nullptr && (*on_final)(i * pl.Cq, pl.Cq) != cudaSuccess)
            return CPATTN_ERR_CUDA;
      }
    } else {
      // Work items keep the ring's launch order; a Pass-KV accumulator
      // update waits (bounded) until the previous visit of the same rows has
      // finished.
      int total = 0;
      double vis = 0.0;
      std::vector<int> visits(pl.P, 0);
      for (auto &pd : table) {
        pd.n_qtiles = (pd.q_len + sh.rows - 1) / sh.rows;
        pd.cta_begin = total;
        total += pd.n_qtiles * per_tile;
        vis += visible_pairs(pd.delta, pd.q_len, 0, pd.kv_len, causal != 0);
        const int piece = (int)(pd.q_row0 / pl.Cq);
        if (pd.mode == kAccInit || pd.mode == kAccMerge || pd.mode == kAccFinal)
          pd.visit = visits[piece]++;
      }
      // Inputs arriving piece by piece: the one launch reads all of them.
      for (int i = 0; i < pl.P && on_inputs != nullptr; ++i)
        if ((*on_inputs)(i, 0) != cudaSuccess) return CPATTN_ERR_CUDA;
      if ((s = launch_table(table, total, vis)) != CPATTN_OK) return s;
    }
  }
  const bool per_step = !(single && attn_tc_supported(p));
  // Pass-Q merge of partials, and empty rows of chunks no key reaches: one
  // launch for the listed pieces.
  MergeNParams mp;
  memset(&mp, 0, sizeof(mp));
  mp.B = (int32_t)q->b;
  mp.H = (int32_t)q->h;
  mp.D = (int32_t)q->d;
  mp.chunk_rows = (int32_t)pl.Cq;
  mp.out = p.out;
  mp.part = p.part;
  mp.part_o_stride = p.part_o_stride;
  mp.part_lse_stride = p.part_lse_stride;
  mp.n_part_slots = pl.n_slots;
  const double row_bytes = (double)q->b * pl.Cq * q->h * (q->d * 4.0 + 4.0);
  const double out_bytes = (double)q->b * pl.Cq * q->h * (q->d * elem_bytes(o->dtype) + 4.0);
  auto needs_merge_launch = [&](int i) {
    return (pl.mode == CPATTN_PASS_Q && pl.count[i] >= 2) || pl.count[i] == 0;
  };
  auto merge_pieces = [&](std::vector<int> pieces) -> cpattn_status {
    // Items with the most partials first (longest CTAs first).
    std::stable_sort(pieces.begin(), pieces.end(),
                     [&](int a, int b) { return pl.count[a] > pl.count[b]; });
    mp.n_items = 0;
    double bytes = 0.0;
    for (int i : pieces) {
      const bool merge = pl.count[i] >= 2;
      mp.item_row0[mp.n_items] = (int32_t)(i * pl.Cq);
      mp.item_slot0[mp.n_items] = merge ? pl.slot0[i] : 0;
      mp.item_count[mp.n_items] = merge ? pl.count[i] : 0;
      bytes += (merge ? pl.count[i] * row_bytes : 0.0) + out_bytes;
      ++mp.n_items;
    }
    if (mp.n_items == 0) return CPATTN_OK;
    NvtxRange range("cpattn %s merge", mode_name(mode));
    prof_before(st);
    cudaError_t e = launch_merge_n(mp, st);
    prof_after(st, CPATTN_KERNEL_MERGEN, bytes);
    if (e != cudaSuccess) return CPATTN_ERR_CUDA;
    for (int i : pieces)
      if (per_step && on_final != nullptr && (*on_final)(i * pl.Cq, pl.Cq) != cudaSuccess)
        return CPATTN_ERR_CUDA;
    return CPATTN_OK;
  };
  // With a finality callback, a piece's Pass-Q merge runs right after the
  // launch that produced its last partial, so its rows can leave early.
  std::vector<int> last_launch(pl.P, -1);
  for (const auto &e : pl.entries)
    if (e.role == CPATTN_ROLE_PARTIAL) last_launch[e.q_chunk] = std::max(last_launch[e.q_chunk], e.launch);
  std::vector<bool> merged(pl.P, false);

  p.persistent_ctas = lmode == CPATTN_LAUNCH_PERSISTENT_STEP ? 1 : 0;
  // Host-buffer Pass-Q calls with long items: every Q piece completes only at
  // the ring's last step, so merges and output copies would all wait for the
  // end.  They run the ring's pairs grouped by Q piece instead (the groups of
  // piece_groups, in arrival order): each pair is computed exactly as in its
  // ring step and each piece is merged in the same order, so the result is
  // the same bit for bit, but a group's merge and output copy overlap the
  // later groups.
  const bool q_grouped = per_step && pl.mode == CPATTN_PASS_Q && on_inputs != nullptr &&
                         on_final != nullptr && !short_items(pl, q_base, causal);
  if (q_grouped) {
    for (const auto &grp : piece_groups(pl.P, true)) {
      NvtxRange range("cpattn %s pieces %d..%d", mode_name(mode), grp.front(), grp.back());
      std::vector<bool> in(pl.P, false);
      for (int i : grp) in[i] = true;
      std::vector<size_t> idx;
      for (size_t x = 0; x < pl.entries.size(); ++x)
        if (in[pl.entries[x].q_chunk]) idx.push_back(x);
      std::vector<PairDesc> items;
      launch_items_of(idx, items);
      for (int i : grp)
        if ((*on_inputs)(i, 0) != cudaSuccess) return CPATTN_ERR_CUDA;
      for (size_t x0 = 0; x0 < items.size(); x0 += kMaxPairs) {
        const size_t n = std::min<size_t>(kMaxPairs, items.size() - x0);
        p.n_pairs = (int32_t)n;
        for (size_t x = 0; x < n; ++x) p.pairs[x] = items[x0 + x];
        if (launch_attn(p, st, q) != cudaSuccess) return CPATTN_ERR_CUDA;
      }
      std::vector<int> ready;
      for (int i : grp) {
        if (needs_merge_launch(i)) {
          ready.push_back(i);
          merged[i] = true;
        } else if ((*on_final)(i * pl.Cq, pl.Cq) != cudaSuccess) {  // one pair: stored directly
          return CPATTN_ERR_CUDA;
        }
      }
      if ((s = merge_pieces(ready)) != CPATTN_OK) return s;
    }
  }

  // One launch per ring step (two per step for zigzag Pass-KV, one per
  // visiting K/V piece).
  size_t e0 = 0;
  for (int l = 0; l < pl.n_launches && per_step && !q_grouped; ++l) {
    size_t e1 = e0;
    while (e1 < pl.entries.size() && pl.entries[e1].launch == l) ++e1;
    if (e1 == e0) continue;
    NvtxRange range("cpattn %s step %d", mode_name(mode), pl.entries[e0].step);
    std::vector<PairDesc> items;
    launch_items(e0, e1, items);
    if (on_inputs != nullptr && l == 0) {
      // Inputs arrive piece by piece: the first ring step runs one pair per
      // launch, each as soon as its pieces are in (its pairs touch disjoint
      // output rows, so splitting the launch changes no arithmetic).
      for (const PairDesc &pd : items) {
        if ((*on_inputs)(pd.q_row0 / (int32_t)pl.Cq, pd.kv_row0 / (int32_t)pl.C) != cudaSuccess)
          return CPATTN_ERR_CUDA;
        p.n_pairs = 1;
        p.pairs[0] = pd;
        if (launch_attn(p, st, q) != cudaSuccess) return CPATTN_ERR_CUDA;
      }
    } else {
      for (const PairDesc &pd : items)
        if (on_inputs != nullptr &&
            (*on_inputs)(pd.q_row0 / (int32_t)pl.Cq, pd.kv_row0 / (int32_t)pl.C) != cudaSuccess)
          return CPATTN_ERR_CUDA;
      p.n_pairs = (int32_t)items.size();
      for (size_t x = 0; x < items.size(); ++x) p.pairs[x] = items[x];
      if (launch_attn(p, st, q) != cudaSuccess) return CPATTN_ERR_CUDA;
    }
    if (on_final != nullptr) {
      std::vector<int> ready;
      for (size_t x = e0; x < e1; ++x) {
        const cpattn_plan_entry &e = pl.entries[x];
        if (e.role == CPATTN_ROLE_STORE || e.role == CPATTN_ROLE_ACC_FINAL) {
          if ((*on_final)(e.q_chunk * pl.Cq, pl.Cq) != cudaSuccess) return CPATTN_ERR_CUDA;
        } else if (e.role == CPATTN_ROLE_PARTIAL && last_launch[e.q_chunk] == l &&
                   needs_merge_launch(e.q_chunk) && !merged[e.q_chunk]) {
          ready.push_back(e.q_chunk);
          merged[e.q_chunk] = true;
        }
      }
      if ((s = merge_pieces(ready)) != CPATTN_OK) return s;
    }
    e0 = e1;
  }

  std::vector<int> rest;
  for (int i = 0; i < pl.P; ++i)
    if (needs_merge_launch(i) && !merged[i]) rest.push_back(i);
  if ((s = merge_pieces(rest)) != CPATTN_OK) return s;
  if (!per_step && on_final != nullptr) {
    if (grouped) {
      // Rows of pieces no key reaches (written by the merge launch above).
      for (int i : rest)
        if ((*on_final)(i * pl.Cq, pl.Cq) != cudaSuccess) return CPATTN_ERR_CUDA;
    } else if ((*on_final)(0, q->s) != cudaSuccess) {
      return CPATTN_ERR_CUDA;
    }
  }
  return CPATTN_OK;
}

// ----------------------------------------------------------------- decode
// Pass-Q decode: n_tok query tokens (the same Q on every emulated CP rank)
// against n_chunks KV chunks.  Every rank splits the part of its chunk that a
// token can see into kv_split-key pieces; each piece yields an fp32 partial,
// and all partials are merged by LSE in ascending (chunk, piece) order.
struct DecodePlan {
  int64_t C = 0;
  int kv_split = 0;
  bool packed = false;              // tensor-core kernel with GQA-packed rows
  std::vector<int> chunk, vis, slot0;  // visible chunks, visible keys, first slot
  int n_slots = 0;
};

constexpr int64_t kDecodeTargetCtas = 1024;  // pieces x kv heads x batch per launch

bool decode_packed_ok(const cpattn_tensor *q, const cpattn_tensor *k) {
  if (q->dtype != CPATTN_BF16 || q->d != 128 || k->s == 0) return false;
  const int64_t g = q->h / k->h;
  return 128 % g == 0 && q->s <= 128 / g;
}

cpattn_status build_decode_plan(const cpattn_tensor *q, const cpattn_tensor *k, int64_t q_base,
                                int n_chunks, int causal, DecodePlan &dp) {
  if (n_chunks < 1 || n_chunks > kMaxPairs) return CPATTN_ERR_INVALID_ARG;
  if (k->s % n_chunks != 0) return CPATTN_ERR_INVALID_ARG;
  if (q_base < -kMaxRows * 4 || q_base > kMaxRows * 4) return CPATTN_ERR_UNSUPPORTED;
  dp.C = k->s / n_chunks;
  dp.packed = decode_packed_ok(q, k);
  int64_t total = 0;
  for (int j = 0; j < n_chunks && q->s > 0 && dp.C > 0; ++j) {
    int64_t vis = dp.C;
    if (causal) {
      const int64_t last = q_base + q->s - 1 - (int64_t)j * dp.C + 1;  // keys the last token sees
      vis = last < 0 ? 0 : (last < dp.C ? last : dp.C);
    }
    if (vis == 0) continue;
    dp.chunk.push_back(j);
    dp.vis.push_back((int)vis);
    total += vis;
  }
  if (dp.packed) {
    int64_t want = (total * k->h * q->b + kDecodeTargetCtas - 1) / kDecodeTargetCtas;
    want = (want + 127) / 128 * 128;
    dp.kv_split = (int)std::min<int64_t>(std::max<int64_t>(want, 256), 65536);
  } else {
    dp.kv_split = (int)std::max<int64_t>(dp.C, 1);  // one piece per chunk
  }
  dp.n_slots = 0;
  for (size_t x = 0; x < dp.chunk.size(); ++x) {
    dp.slot0.push_back(dp.n_slots);
    dp.n_slots += (dp.vis[x] + dp.kv_split - 1) / dp.kv_split;
  }
  return CPATTN_OK;
}

size_t decode_ws_bytes(const DecodePlan &dp, const cpattn_tensor *q) {
  const size_t o = (size_t)dp.n_slots * q->b * q->s * q->h * q->d * 4;
  const size_t l = (size_t)dp.n_slots * q->b * q->h * q->s * 4;
  return align256(o) + align256(l);
}

size_t tensor_bytes(const cpattn_tensor *t) {
  return (size_t)t->b * t->s * t->h * t->d * elem_bytes(t->dtype);
}

bool is_contiguous(const cpattn_tensor *t) {
  return t->stride_h == t->d && t->stride_s == t->h * t->d &&
         (t->b == 1 || t->stride_b == t->s * t->h * t->d);
}

cpattn_tensor dense_like(const cpattn_tensor *t, void *data, int32_t dtype) {
  cpattn_tensor r = *t;
  r.data = data;
  r.dtype = dtype;
  r.stride_h = t->d;
  r.stride_s = t->h * t->d;
  r.stride_b = t->s * t->h * t->d;
  return r;
}

}  // namespace

extern "C" {

const char *cpattn_status_string(cpattn_status s) {
  switch (s) {
    case CPATTN_OK: return "CPATTN_OK";
    case CPATTN_ERR_INVALID_ARG: return "CPATTN_ERR_INVALID_ARG: bad argument";
    case CPATTN_ERR_UNSUPPORTED: return "CPATTN_ERR_UNSUPPORTED: shape or dtype not supported";
    case CPATTN_ERR_WORKSPACE: return "CPATTN_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case CPATTN_ERR_CUDA: return "CPATTN_ERR_CUDA: a CUDA call or launch failed";
    case CPATTN_ERR_TIMEOUT: return "CPATTN_ERR_TIMEOUT: a kernel-side wait gave up";
    case CPATTN_ERR_DEVICE_CHECK:
      return "CPATTN_ERR_DEVICE_CHECK: a debug-build kernel bounds check failed";
  }
  return "CPATTN: unknown status";
}

cpattn_status cpattn_partial(const cpattn_tensor *q, const cpattn_tensor *k,
                             const cpattn_tensor *v, int64_t q_off, int64_t kv_off, int causal,
                             float scale, cpattn_tensor *o, float *lse, void *stream) {
  try {
    cpattn_status s = check_qkv(q, k, v);
    if (s != CPATTN_OK) return s;
    if ((s = check_out(o, lse, q)) != CPATTN_OK) return s;
    if (q_off < -kMaxRows * 4 || q_off > kMaxRows * 4 || kv_off < -kMaxRows * 4 ||
        kv_off > kMaxRows * 4)
      return CPATTN_ERR_UNSUPPORTED;
    if (q->s == 0) return CPATTN_OK;
    NvtxRange range("cpattn partial");
    AttnParams p;
    fill_inputs(p, q, k, v, causal, scale);
    p.out = out_view(o, lse);
    p.n_pairs = 1;
    p.pairs[0].q_row0 = 0;
    p.pairs[0].q_len = (int32_t)q->s;
    p.pairs[0].kv_row0 = 0;
    p.pairs[0].kv_len = (int32_t)k->s;
    p.pairs[0].delta = q_off - kv_off;
    p.pairs[0].mode = kStore;
    p.pairs[0].slot = -1;
    return launch_attn(p, reinterpret_cast<cudaStream_t>(stream), q) == cudaSuccess
               ? CPATTN_OK
               : CPATTN_ERR_CUDA;
  } catch (...) {
    return CPATTN_ERR_INVALID_ARG;
  }
}

cpattn_status cpattn_merge(cpattn_tensor *o_a, float *lse_a, const cpattn_tensor *o_b,
                           const float *lse_b, void *stream) {
  cpattn_status s = check_view(o_a);
  if (s != CPATTN_OK) return s;
  if ((s = check_view(o_b)) != CPATTN_OK) return s;
  if (o_a->dtype != o_b->dtype || o_a->b != o_b->b || o_a->s != o_b->s || o_a->h != o_b->h ||
      o_a->d != o_b->d)
    return CPATTN_ERR_INVALID_ARG;
  if (o_a->d != 64 && o_a->d != 128) return CPATTN_ERR_UNSUPPORTED;
  if (o_a->s > 0 && (lse_a == nullptr || lse_b == nullptr)) return CPATTN_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(lse_a) % 4 || reinterpret_cast<uintptr_t>(lse_b) % 4)
    return CPATTN_ERR_INVALID_ARG;
  if (o_a->s == 0) return CPATTN_OK;
  Merge2Params p;
  memset(&p, 0, sizeof(p));
  p.B = (int32_t)o_a->b;
  p.S = (int32_t)o_a->s;
  p.H = (int32_t)o_a->h;
  p.D = (int32_t)o_a->d;
  p.a = out_view(o_a, lse_a);
  p.b = out_view(o_b, const_cast<float *>(lse_b));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  NvtxRange range("cpattn merge");
  const double bytes = 3.0 * (double)o_a->b * o_a->s * o_a->h * (o_a->d * elem_bytes(o_a->dtype) + 4.0);
  prof_before(st);
  cudaError_t e = launch_merge_2(p, st);
  prof_after(st, CPATTN_KERNEL_MERGE2, bytes);
  return e == cudaSuccess ? CPATTN_OK : CPATTN_ERR_CUDA;
}

cpattn_status cpattn_prefill_workspace_size(const cpattn_tensor *q, const cpattn_tensor *k,
                                            int64_t q_base, int n_chunks, int mode, int causal,
                                            size_t *bytes) {
  return cpattn_prefill_workspace_size_ex(q, k, q_base, n_chunks, mode, causal, nullptr, bytes);
}

static cpattn_status prefill_ws_bytes(const cpattn_tensor *q, const cpattn_tensor *k, int64_t q_base,
                               int n_chunks, int mode, int causal,
                               const cpattn_prefill_options *opts, size_t *bytes) {
  try {
    if (bytes == nullptr) return CPATTN_ERR_INVALID_ARG;
    cpattn_status s = check_view(q);
    if (s != CPATTN_OK) return s;
    if ((s = check_view(k)) != CPATTN_OK) return s;
    Plan pl;
    if ((s = build_plan(q->s, k->s, q_base, n_chunks, mode, causal, assignment_of(opts), pl)) !=
        CPATTN_OK)
      return s;
    if (!valid_launch(launch_mode_of(opts))) return CPATTN_ERR_INVALID_ARG;
    const int lmode = resolve_launch(launch_mode_of(opts), pl, q, k, q_base, causal);
    *bytes = ws_layout(pl, q->b, q->s, q->h, q->d, lmode).total;
    return CPATTN_OK;
  } catch (...) {
    return CPATTN_ERR_INVALID_ARG;
  }
}

cpattn_status cpattn_prefill_workspace_size_ex(const cpattn_tensor *q, const cpattn_tensor *k,
                                               int64_t q_base, int n_chunks, int mode, int causal,
                                               const cpattn_prefill_options *opts, size_t *bytes) {
  return prefill_ws_bytes(q, k, q_base, n_chunks, mode, causal, opts, bytes);
}

cpattn_status cpattn_prefill_launch_mode(const cpattn_tensor *q, const cpattn_tensor *k,
                                         int64_t q_base, int n_chunks, int mode, int causal,
                                         const cpattn_prefill_options *opts, int *launch) {
  try {
    if (launch == nullptr) return CPATTN_ERR_INVALID_ARG;
    cpattn_status s = check_view(q);
    if (s != CPATTN_OK) return s;
    if ((s = check_view(k)) != CPATTN_OK) return s;
    const int lmode = launch_mode_of(opts);
    if (!valid_launch(lmode)) return CPATTN_ERR_INVALID_ARG;
    Plan pl;
    if ((s = build_plan(q->s, k->s, q_base, n_chunks, mode, causal, assignment_of(opts), pl)) !=
        CPATTN_OK)
      return s;
    *launch = resolve_launch(lmode, pl, q, k, q_base, causal);
    return CPATTN_OK;
  } catch (...) {
    return CPATTN_ERR_INVALID_ARG;
  }
}

cpattn_status cpattn_prefill(const cpattn_tensor *q, const cpattn_tensor *k,
                             const cpattn_tensor *v, int64_t q_base, int n_chunks, int mode,
                             int causal, float scale, cpattn_tensor *o, float *lse,
                             void *workspace, size_t workspace_bytes, void *stream) {
  return cpattn_prefill_ex(q, k, v, q_base, n_chunks, mode, causal, scale, o, lse, workspace,
                           workspace_bytes, nullptr, stream);
}

cpattn_status cpattn_prefill_ex(const cpattn_tensor *q, const cpattn_tensor *k,
                                const cpattn_tensor *v, int64_t q_base, int n_chunks, int mode,
                                int causal, float scale, cpattn_tensor *o, float *lse,
                                void *workspace, size_t workspace_bytes,
                                const cpattn_prefill_options *opts, void *stream) {
  try {
    return prefill_impl(q, k, v, q_base, n_chunks, mode, causal, scale, o, lse, workspace,
                        workspace_bytes, opts, reinterpret_cast<cudaStream_t>(stream));
  } catch (...) {
    return CPATTN_ERR_INVALID_ARG;
  }
}

cpattn_status cpattn_decode_workspace_size(const cpattn_tensor *q, const cpattn_tensor *k,
                                           int64_t q_base, int n_chunks, int causal,
                                           size_t *bytes) {
  try {
    if (bytes == nullptr) return CPATTN_ERR_INVALID_ARG;
    cpattn_status s = check_view(q);
    if (s != CPATTN_OK) return s;
    if ((s = check_view(k)) != CPATTN_OK) return s;
    if (q->h % k->h != 0) return CPATTN_ERR_INVALID_ARG;
    DecodePlan dp;
    if ((s = build_decode_plan(q, k, q_base, n_chunks, causal, dp)) != CPATTN_OK) return s;
    *bytes = decode_ws_bytes(dp, q);
    return CPATTN_OK;
  } catch (...) {
    return CPATTN_ERR_INVALID_ARG;
  }
}

cpattn_status cpattn_decode(const cpattn_tensor *q, const cpattn_tensor *k, const cpattn_tensor *v,
                            int64_t q_base, int n_chunks, int causal, float scale,
                            cpattn_tensor *o, float *lse, void *workspace, size_t workspace_bytes,
                            void *stream) {
  try {
    cpattn_status s = check_qkv(q, k, v);
    if (s != CPATTN_OK) return s;
    if ((s = check_out(o, lse, q)) != CPATTN_OK) return s;
    DecodePlan dp;
    if ((s = build_decode_plan(q, k, q_base, n_chunks, causal, dp)) != CPATTN_OK) return s;
    const size_t need = decode_ws_bytes(dp, q);
    if (dp.n_slots > 0) {
      if (workspace == nullptr || workspace_bytes < need) return CPATTN_ERR_WORKSPACE;
      if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return CPATTN_ERR_WORKSPACE;
    }
    if (q->s == 0) return CPATTN_OK;
    NvtxRange range("cpattn decode");
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *ws = reinterpret_cast<uint8_t *>(workspace);
    AttnParams p;
    fill_inputs(p, q, k, v, causal, scale);
    p.out = out_view(o, lse);
    if (dp.n_slots > 0) {
      const size_t o_bytes = (size_t)dp.n_slots * q->b * q->s * q->h * q->d * 4;
      p.part.o = ws;
      p.part.lse = reinterpret_cast<float *>(ws + align256(o_bytes));
      p.part.sh = q->d;
      p.part.ss = q->h * q->d;
      p.part.sb = q->s * q->h * q->d;
      p.part.lh = q->s;
      p.part.lb = q->h * q->s;
      p.part.f32 = 1;
      p.part_o_stride = q->b * q->s * q->h * q->d;
      p.part_lse_stride = q->b * q->h * q->s;
      p.n_part_slots = dp.n_slots;
      p.part_rows = (int32_t)q->s;
      p.n_pairs = (int32_t)dp.chunk.size();
      for (size_t x = 0; x < dp.chunk.size(); ++x) {
        PairDesc &pd = p.pairs[x];
        pd.q_row0 = 0;
        pd.q_len = (int32_t)q->s;
        pd.kv_row0 = (int32_t)(dp.chunk[x] * dp.C);
        pd.kv_len = dp.vis[x];
        pd.delta = q_base - (int64_t)dp.chunk[x] * dp.C;
        pd.mode = kPartial;
        pd.slot = dp.slot0[x];
      }
      if (dp.packed) {
        p.pack_g = (int32_t)(q->h / k->h);
        p.kv_split = dp.kv_split;
        p.persistent_ctas = 1;  // many short items: loop over them, one CTA per SM
      }
      if (launch_attn(p, st, q) != cudaSuccess) return CPATTN_ERR_CUDA;
    }
    MergeNParams mp;
    memset(&mp, 0, sizeof(mp));
    mp.B = (int32_t)q->b;
    mp.H = (int32_t)q->h;
    mp.D = (int32_t)q->d;
    mp.chunk_rows = (int32_t)q->s;
    mp.out = p.out;
    mp.part = p.part;
    mp.part_o_stride = p.part_o_stride;
    mp.part_lse_stride = p.part_lse_stride;
    mp.n_items = 1;
    mp.item_row0[0] = 0;
    mp.item_slot0[0] = 0;
    mp.item_count[0] = dp.n_slots;
    mp.n_part_slots = dp.n_slots;
    const double bytes = (double)dp.n_slots * q->b * q->s * q->h * (q->d * 4.0 + 4.0) +
                         (double)q->b * q->s * q->h * (q->d * elem_bytes(o->dtype) + 4.0);
    prof_before(st);
    cudaError_t e = launch_merge_n(mp, st);
    prof_after(st, CPATTN_KERNEL_MERGEN, bytes);
    return e == cudaSuccess ? CPATTN_OK : CPATTN_ERR_CUDA;
  } catch (...) {
    return CPATTN_ERR_INVALID_ARG;
  }
}

cpattn_status cpattn_prefill_choose_mode(const cpattn_tensor *q, const cpattn_tensor *k,
                                         int n_chunks, int *mode, double *pass_kv_bytes,
                                         double *pass_q_bytes) {
  if (mode == nullptr || q == nullptr || k == nullptr) return CPATTN_ERR_INVALID_ARG;
  const int es = elem_bytes(q->dtype);
  if (es == 0 || n_chunks < 1 || q->h < 1 || k->h < 1 || q->d < 1) return CPATTN_ERR_INVALID_ARG;
  const double N = n_chunks, hops = N * (N - 1);
  const double ckv = (double)k->s / N, cq = (double)q->s / N;
  const double kv = hops * 2.0 * ckv * (double)k->h * (double)q->d * es * (double)q->b;
  const double qb = hops * cq * (double)q->h * ((double)q->d * es * 2.0 + 4.0) * (double)q->b;
  *mode = qb < kv ? CPATTN_PASS_Q : CPATTN_PASS_KV;
  if (pass_kv_bytes) *pass_kv_bytes = kv;
  if (pass_q_bytes) *pass_q_bytes = qb;
  return CPATTN_OK;
}

cpattn_status cpattn_prefill_choose_mode_ex(const cpattn_tensor *q, const cpattn_tensor *k,
                                            int64_t q_base, int n_chunks, int causal,
                                            const cpattn_prefill_options *opts, int *mode,
                                            double *pass_kv_bytes, double *pass_q_bytes) {
  try {
    if (mode == nullptr || q == nullptr || k == nullptr) return CPATTN_ERR_INVALID_ARG;
    const int es = elem_bytes(q->dtype);
    if (es == 0 || q->h < 1 || k->h < 1 || q->d < 1 || q->b < 1) return CPATTN_ERR_INVALID_ARG;
    Plan pl;
    cpattn_status s =
        build_plan(q->s, k->s, q_base, n_chunks, CPATTN_PASS_KV, causal, assignment_of(opts), pl);
    if (s != CPATTN_OK) return s;
    const int N = pl.N;
    const bool cz = causal != 0;
    // need[r * N + s]: some Q piece of rank r sees some K/V piece of rank s.
    std::vector<char> need((size_t)N * N, 0);
    int64_t remote_pairs = 0;  // visible piece pairs whose Q and K/V live on different ranks
    for (int r = 0; r < N; ++r)
      for (int t = 0; t < N; ++t) {
        int qp[2], kp[2];
        const int nq = rank_pieces(pl, r, qp), nk = rank_pieces(pl, t, kp);
        for (int a = 0; a < nq; ++a)
          for (int b = 0; b < nk; ++b)
            if (pair_visible(pl, q_base, cz, qp[a], kp[b])) {
              need[(size_t)r * N + t] = 1;
              if (r != t) ++remote_pairs;
            }
      }
    // A travelling chunk moves one rank per step in the ring's direction (rank
    // r receives the chunk of rank (r - 1) mod N) until the farthest rank that
    // needs it has it.
    const int ppr = pl.P / N;  // pieces per rank
    const double kv_unit = (double)ppr * pl.C * k->h * q->d * es * 2.0 * q->b;
    const double q_unit = (double)ppr * pl.Cq * q->h * q->d * es * (double)q->b;
    const double ret_unit = (double)pl.Cq * q->h * ((double)q->d * es + 4.0) * q->b;
    double kv = 0.0, qb = 0.0;
    for (int t = 0; t < N; ++t) {  // K/V of rank t travel to the ranks whose Q sees them
      int hops = 0;
      for (int r = 0; r < N; ++r)
        if (r != t && need[(size_t)r * N + t]) hops = std::max(hops, ((r - t) % N + N) % N);
      kv += hops * kv_unit;
    }
    for (int r = 0; r < N; ++r) {  // Q of rank r travels to the ranks whose K/V it sees
      int hops = 0;
      for (int t = 0; t < N; ++t)
        if (t != r && need[(size_t)r * N + t]) hops = std::max(hops, ((t - r) % N + N) % N);
      qb += hops * q_unit;
    }
    qb += (double)remote_pairs * ret_unit;  // each remote partial (O, LSE) returns once
    *mode = qb < kv ? CPATTN_PASS_Q : CPATTN_PASS_KV;
    if (pass_kv_bytes) *pass_kv_bytes = kv;
    if (pass_q_bytes) *pass_q_bytes = qb;
    return CPATTN_OK;
  } catch (...) {
    return CPATTN_ERR_INVALID_ARG;
  }
}

cpattn_status cpattn_prefill_plan(int64_t sq, int64_t skv, int64_t q_base, int n_chunks, int mode,
                                  int causal, cpattn_plan_entry *entries, int capacity,
                                  int *n_entries) {
  return cpattn_prefill_plan_ex(sq, skv, q_base, n_chunks, mode, causal, nullptr, entries,
                                capacity, n_entries);
}

cpattn_status cpattn_prefill_critical_path(int64_t sq, int64_t skv, int64_t q_base, int n_chunks,
                                           int mode, int causal,
                                           const cpattn_prefill_options *opts,
                                           double *step_max, double *critical, double *total) {
  try {
    if (critical == nullptr || total == nullptr) return CPATTN_ERR_INVALID_ARG;
    Plan pl;
    cpattn_status s = build_plan(sq, skv, q_base, n_chunks, mode, causal, assignment_of(opts), pl);
    if (s != CPATTN_OK) return s;
    std::vector<double> sm;
    plan_work(pl, q_base, causal != 0, sm, *critical, *total);
    if (step_max)
      for (int t = 0; t < n_chunks; ++t) step_max[t] = sm[t];
    return CPATTN_OK;
  } catch (...) {
    return CPATTN_ERR_INVALID_ARG;
  }
}

cpattn_status cpattn_prefill_plan_ex(int64_t sq, int64_t skv, int64_t q_base, int n_chunks,
                                     int mode, int causal, const cpattn_prefill_options *opts,
                                     cpattn_plan_entry *entries, int capacity, int *n_entries) {
  try {
    if (n_entries == nullptr || capacity < 0 || (capacity > 0 && entries == nullptr))
      return CPATTN_ERR_INVALID_ARG;
    Plan pl;
    cpattn_status s = build_plan(sq, skv, q_base, n_chunks, mode, causal, assignment_of(opts), pl);
    if (s != CPATTN_OK) return s;
    *n_entries = (int)pl.entries.size();
    for (int x = 0; x < capacity && x < (int)pl.entries.size(); ++x) entries[x] = pl.entries[x];
    return CPATTN_OK;
  } catch (...) {
    return CPATTN_ERR_INVALID_ARG;
  }
}

cpattn_status cpattn_prefill_host_scratch_size(const cpattn_tensor *q, const cpattn_tensor *k,
                                               int64_t q_base, int n_chunks, int mode, int causal,
                                               int out_dtype, size_t *bytes) {
  if (bytes == nullptr || elem_bytes(out_dtype) == 0) return CPATTN_ERR_INVALID_ARG;
  size_t ws = 0;
  cpattn_status s = prefill_ws_bytes(q, k, q_base, n_chunks, mode, causal, nullptr, &ws);
  if (s != CPATTN_OK) return s;
  const size_t o_bytes = (size_t)q->b * q->s * q->h * q->d * elem_bytes(out_dtype);
  *bytes = align256(tensor_bytes(q)) + 2 * align256(tensor_bytes(k)) + align256(o_bytes) +
           align256((size_t)q->b * q->h * q->s * 4) + ws;
  return CPATTN_OK;
}

// Side streams and events of one host-buffer call, released on every path out.
struct CopyStream {
  cudaStream_t s = nullptr;
  std::vector<cudaEvent_t> events;
  ~CopyStream() {
    if (s != nullptr) {
      cudaStreamSynchronize(s);
      cudaStreamDestroy(s);
    }
    for (auto ev : events) cudaEventDestroy(ev);
  }
  cudaError_t record(cudaStream_t on, cudaEvent_t *out) {
    cudaError_t e = cudaEventCreateWithFlags(out, cudaEventDisableTiming);
    if (e != cudaSuccess) return e;
    events.push_back(*out);
    return cudaEventRecord(*out, on);
  }
};

cpattn_status cpattn_prefill_host(const cpattn_tensor *q, const cpattn_tensor *k,
                                  const cpattn_tensor *v, int64_t q_base, int n_chunks, int mode,
                                  int causal, float scale, cpattn_tensor *o, float *lse,
                                  void *dev_scratch, size_t scratch_bytes, void *stream) {
  try {
    cpattn_status s = check_qkv(q, k, v);
    if (s != CPATTN_OK) return s;
    if ((s = check_out(o, lse, q)) != CPATTN_OK) return s;
    if (!is_contiguous(q) || !is_contiguous(k) || !is_contiguous(v) || !is_contiguous(o))
      return CPATTN_ERR_INVALID_ARG;
    size_t need = 0;
    if ((s = cpattn_prefill_host_scratch_size(q, k, q_base, n_chunks, mode, causal, o->dtype,
                                              &need)) != CPATTN_OK)
      return s;
    if (dev_scratch == nullptr || scratch_bytes < need ||
        reinterpret_cast<uintptr_t>(dev_scratch) % 256 != 0)
      return CPATTN_ERR_WORKSPACE;
    NvtxRange range("cpattn prefill_host %s", mode_name(mode));
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *base = reinterpret_cast<uint8_t *>(dev_scratch);
    size_t off = 0;
    auto take = [&](size_t n) { uint8_t *r = base + off; off += align256(n); return r; };
    const size_t o_bytes = tensor_bytes(o);
    const size_t lse_bytes = (size_t)q->b * q->h * q->s * 4;
    cpattn_tensor dq = dense_like(q, take(tensor_bytes(q)), q->dtype);
    cpattn_tensor dk = dense_like(k, take(tensor_bytes(k)), k->dtype);
    cpattn_tensor dv = dense_like(v, take(tensor_bytes(v)), v->dtype);
    cpattn_tensor dout = dense_like(o, take(o_bytes), o->dtype);
    float *dlse = reinterpret_cast<float *>(take(lse_bytes));
    void *ws = base + off;
    const size_t ws_bytes = scratch_bytes - off;
    if (q->s == 0) return CPATTN_OK;
    Plan pl;
    if ((s = build_plan(q->s, k->s, q_base, n_chunks, mode, causal, CPATTN_ASSIGN_CONTIGUOUS, pl)) !=
        CPATTN_OK)
      return s;
    // Inputs come in on one side stream (K and V first, then Q a piece at a
    // time) while the first ring step starts on each piece as it lands;
    // output rows go back on another as soon as the launch that finalises
    // them has been enqueued (a Pass-KV piece after its last ring step, a
    // Pass-Q piece after its merge), overlapping both directions of copies
    // with the ring.
    CopyStream up, down;
    if (cudaStreamCreateWithFlags(&up.s, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&down.s, cudaStreamNonBlocking) != cudaSuccess)
      return CPATTN_ERR_CUDA;
    // The caller's stream may hold earlier work on the scratch buffer.
    cudaEvent_t ev_start, ev_kv;
    if (up.record(st, &ev_start) != cudaSuccess || cudaStreamWaitEvent(up.s, ev_start, 0) != cudaSuccess)
      return CPATTN_ERR_CUDA;
    if (cudaMemcpyAsync(dk.data, k->data, tensor_bytes(k), cudaMemcpyHostToDevice, up.s) != cudaSuccess ||
        cudaMemcpyAsync(dv.data, v->data, tensor_bytes(v), cudaMemcpyHostToDevice, up.s) != cudaSuccess ||
        up.record(up.s, &ev_kv) != cudaSuccess)
      return CPATTN_ERR_CUDA;
    const int64_t q_row_bytes = q->h * q->d * elem_bytes(q->dtype);
    std::vector<cudaEvent_t> ev_q(pl.P);
    for (int i = 0; i < pl.P; ++i) {
      if (cudaMemcpy2DAsync(static_cast<uint8_t *>(dq.data) + i * pl.Cq * q_row_bytes,
                            q->s * q_row_bytes,
                            static_cast<const uint8_t *>(q->data) + i * pl.Cq * q_row_bytes,
                            q->s * q_row_bytes, pl.Cq * q_row_bytes, q->b, cudaMemcpyHostToDevice,
                            up.s) != cudaSuccess ||
          up.record(up.s, &ev_q[i]) != cudaSuccess)
        return CPATTN_ERR_CUDA;
    }
    std::vector<bool> have_q(pl.P, false);
    bool have_kv = false;
    const InputsFn on_inputs = [&](int q_piece, int kv_piece) -> cudaError_t {
      (void)kv_piece;
      cudaError_t e = cudaSuccess;
      if (!have_kv && (e = cudaStreamWaitEvent(st, ev_kv, 0)) != cudaSuccess) return e;
      have_kv = true;
      if (q_piece >= 0 && q_piece < pl.P && !have_q[q_piece]) {
        if ((e = cudaStreamWaitEvent(st, ev_q[q_piece], 0)) != cudaSuccess) return e;
        have_q[q_piece] = true;
      }
      return e;
    };
    const int64_t row_bytes = q->h * q->d * elem_bytes(o->dtype);
    const FinalRowsFn on_final = [&](int64_t row0, int64_t rows) -> cudaError_t {
      cudaEvent_t ev;
      cudaError_t e = down.record(st, &ev);
      if (e != cudaSuccess) return e;
      if ((e = cudaStreamWaitEvent(down.s, ev, 0)) != cudaSuccess) return e;
      // O [b, s, h, d]: one block of rows per batch entry.
      e = cudaMemcpy2DAsync(static_cast<uint8_t *>(o->data) + row0 * row_bytes, q->s * row_bytes,
                            static_cast<uint8_t *>(dout.data) + row0 * row_bytes, q->s * row_bytes,
                            rows * row_bytes, q->b, cudaMemcpyDeviceToHost, down.s);
      if (e != cudaSuccess) return e;
      // LSE [b, h, s]: one run of rows per (batch, head).
      return cudaMemcpy2DAsync(lse + row0, q->s * 4, dlse + row0, q->s * 4, rows * 4, q->b * q->h,
                               cudaMemcpyDeviceToHost, down.s);
    };
    s = prefill_impl(&dq, &dk, &dv, q_base, n_chunks, mode, causal, scale, &dout, dlse, ws,
                     ws_bytes, nullptr, st, &on_final, &on_inputs);
    if (s != CPATTN_OK) return s;
    // Rows no launch reads (a piece no key reaches) still wait for every input.
    for (int i = 0; i < pl.P; ++i)
      if (on_inputs(i, 0) != cudaSuccess) return CPATTN_ERR_CUDA;
    if (cudaStreamSynchronize(down.s) != cudaSuccess) return CPATTN_ERR_CUDA;
    return cudaStreamSynchronize(st) == cudaSuccess ? CPATTN_OK : CPATTN_ERR_CUDA;
  } catch (...) {
    return CPATTN_ERR_INVALID_ARG;
  }
}

cpattn_status cpattn_device_status(int clear) {
  if (cudaDeviceSynchronize() != cudaSuccess) return CPATTN_ERR_CUDA;
  unsigned int (*readers[])(bool, cudaError_t *) = {attn_tc_read_status, attn_pair_read_status,
                                                     attn_simt_read_status, merge_read_status};
  unsigned int v = 0;
  for (auto rd : readers) {
    cudaError_t e = cudaSuccess;
    v |= rd(clear != 0, &e);
    if (e != cudaSuccess) return CPATTN_ERR_CUDA;
  }
  if (v & kStatusTimeout) return CPATTN_ERR_TIMEOUT;
  return (v & kStatusBounds) ? CPATTN_ERR_DEVICE_CHECK : CPATTN_OK;
}

cpattn_status cpattn_profile_begin(int capacity) {
  try {
    if (capacity < 1 || g_prof.armed) return CPATTN_ERR_INVALID_ARG;
    g_prof.events.assign(2 * capacity, nullptr);
    for (auto &ev : g_prof.events)
      if (cudaEventCreate(&ev) != cudaSuccess) return CPATTN_ERR_CUDA;
    g_prof.kinds.assign(capacity, 0);
    g_prof.work.assign(capacity, 0.0);
    g_prof.capacity = capacity;
    g_prof.n = 0;
    g_prof.armed = true;
    return CPATTN_OK;
  } catch (...) {
    return CPATTN_ERR_INVALID_ARG;
  }
}

cpattn_status cpattn_profile_end(cpattn_profile_record *records, int capacity, int *n_records) {
  if (!g_prof.armed) return CPATTN_ERR_INVALID_ARG;
  cpattn_status s = CPATTN_OK;
  const int n = g_prof.n;
  if (n_records) *n_records = n;
  if (n > 0 && cudaEventSynchronize(g_prof.events[2 * n - 1]) != cudaSuccess) s = CPATTN_ERR_CUDA;
  for (int x = 0; x < n && x < capacity && records && s == CPATTN_OK; ++x) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, g_prof.events[2 * x], g_prof.events[2 * x + 1]) != cudaSuccess)
      s = CPATTN_ERR_CUDA;
    records[x].kind = g_prof.kinds[x];
    records[x].ms = ms;
    records[x].work = g_prof.work[x];
  }
  for (auto ev : g_prof.events)
    if (ev) cudaEventDestroy(ev);
  g_prof.events.clear();
  g_prof.armed = false;
  g_prof.n = 0;
  return s;
}

}  // extern "C"
