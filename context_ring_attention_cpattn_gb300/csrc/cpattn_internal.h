// Internal structures shared by the C ABI layer (api.cu) and the kernels.
// Nothing here is part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "cpattn.h"

namespace cpattn {

constexpr int kMaxPairs = 64;  // pairs per launch = ranks per ring step (n_chunks <= 64)

// Debug builds (-DCPATTN_DEBUG) check, in every kernel, each destination row,
// workspace slot and progress counter against its extent before the write; a
// failed check skips the write and sets kStatusBounds in the kernel's device
// status word (cpattn_device_status -> CPATTN_ERR_DEVICE_CHECK).  No check
// traps.
#ifdef CPATTN_DEBUG
constexpr bool kDebugChecks = true;
#else
constexpr bool kDebugChecks = false;
#endif
constexpr unsigned int kStatusTimeout = 1u;  // a bounded wait gave up
constexpr unsigned int kStatusBounds = 2u;   // a debug-build bounds check failed

// Where a pair's result goes (mirrors cpattn_role).
enum PairMode : int32_t {
  kStore = CPATTN_ROLE_STORE,
  kAccInit = CPATTN_ROLE_ACC_INIT,
  kAccMerge = CPATTN_ROLE_ACC_MERGE,
  kAccFinal = CPATTN_ROLE_ACC_FINAL,
  kPartial = CPATTN_ROLE_PARTIAL,
};

// A strided [b, s, h, d] output view plus its LSE [b, h, s] view.
struct OutView {
  void *o;          // bf16 or fp32
  float *lse;
  int64_t sb, ss, sh;  // element strides of o
  int64_t lb, lh;      // element strides of lse (row stride 1)
  int32_t f32;         // 1: o is fp32, 0: bf16
  int32_t pad;
};

// One (Q-chunk, KV-chunk) pair of a launch.
struct PairDesc {
  int32_t q_row0, q_len;    // query rows [q_row0, q_row0 + q_len) of the q tensor
  int32_t kv_row0, kv_len;  // key rows [kv_row0, kv_row0 + kv_len) of k/v
  int64_t delta;            // absolute position of q_row0 minus that of kv_row0
  int32_t mode;             // PairMode
  int32_t slot;             // kPartial: workspace slot index
  int32_t cta_begin;        // filled by the launcher: first work item of this pair
  int32_t n_qtiles;         // filled by the launcher
  int32_t visit;            // Pass-KV, one launch for all steps: visits of this Q piece before
  int32_t dep_base;         // ... and the base of its progress counters
};

struct AttnParams {
  int32_t B, Hq, Hkv, D;
  int32_t causal, n_pairs;
  float scale;              // logit scale
  float scale_log2;         // scale * log2(e)
  // Raw views of the inputs (the SIMT kernel reads them directly; the tensor
  // core kernel uses TMA descriptors built from the same views).
  const void *q, *k, *v;
  int64_t q_sb, q_ss, q_sh, k_sb, k_ss, k_sh, v_sb, v_ss, v_sh;
  int64_t q_rows_total, kv_rows_total;  // s extent of the q and k/v tensors
  int32_t in_f32;           // inputs are fp32 (else bf16)
  int32_t total_ctas;       // filled by the launcher
  // Decode layout (tensor-core kernel only): pack_g > 0 packs the pack_g
  // query heads that share a kv head, for up to 128 / pack_g query rows, into
  // one 128-row tile (tile row r = row r / pack_g, head hk * pack_g + r % pack_g),
  // and each CTA takes kv_split keys of its pair, writing an fp32 partial to
  // slot pairs[x].slot + split.  pack_g = 0: one head per tile row block.
  int32_t pack_g;
  // Per-head tiles (pack_g == 0) with an odd group size Hq / Hkv: a work item
  // is two consecutive 128-row query tiles of one head (which share every K/V
  // tile) instead of one 128-row tile of two heads (filled by the launcher).
  int32_t row_pair;
  int32_t kv_split;
  // Work items: pairs[] (at most kMaxPairs) or, when pair_table is set, a
  // device-resident table of n_table pairs (all ring steps of one call).
  const PairDesc *pair_table;
  int32_t n_table;
  // Grid size for a persistent launch (each CTA loops over work items); 0 =
  // one CTA per work item.
  int32_t persistent_ctas;
  // Pass-KV in one launch: per (Q-piece tile, head, batch) count of warps
  // that finished an accumulator update (4 per update); an update waits until
  // the count reaches 4 * its visit (+ dep_hold, nonzero only to make the
  // bounded wait run out when testing failure detection).
  int32_t *dep_counters;
  int32_t dep_hold;
  // Bound of every kernel-side wait, in ns of global time (set by the
  // launcher from the launch's planned work; at least 2 s).
  uint64_t wait_ns;
  // Extents for the debug-build bounds checks: workspace slots and rows per
  // slot of `part`, and the number of progress counters.
  int32_t n_part_slots, part_rows, n_dep_counters;
  // Nonzero: pair_table groups the pairs of each query piece (ring order)
  // into one run of work items that accumulates on chip (attn_pair only).
  int32_t seg_groups;
  OutView out;              // final output (absolute q rows)
  OutView acc;              // Pass-KV fp32 accumulator (absolute q rows)
  OutView part;             // Pass-Q slot 0 (chunk-relative rows)
  int64_t part_o_stride;    // elements between slots
  int64_t part_lse_stride;
  PairDesc pairs[kMaxPairs];
};

// N-way merge of Pass-Q partials: for each listed Q chunk, merge `count`
// consecutive slots starting at `slot0` (ascending KV chunk) into `out`.
struct MergeNParams {
  int32_t B, H, D, chunk_rows;
  int32_t n_items;
  int32_t n_part_slots;  // slots of `part` (debug-build bounds checks)
  OutView out;
  OutView part;
  int64_t part_o_stride, part_lse_stride;
  int32_t item_row0[kMaxPairs];   // absolute first q row of the chunk
  int32_t item_slot0[kMaxPairs];
  int32_t item_count[kMaxPairs];  // 0 => empty rows (O = 0, LSE = -inf)
};

// Pairwise in-place merge.
struct Merge2Params {
  int32_t B, S, H, D;
  OutView a;   // in/out
  OutView b;
};

// Launchers (return cudaSuccess or the launch error).
//   launch_attn_tc     tensor-core kernels: per-head tiles (pack_g == 0) on a
//                      CTA pair (attn_pair.cu), packed decode tiles
//                      (pack_g > 0) on one CTA (attn_tc.cu)
cudaError_t launch_attn_tc(AttnParams &p, cudaStream_t stream);
cudaError_t launch_attn_pair(AttnParams &p, cudaStream_t stream);
cudaError_t launch_attn_decode_tc(AttnParams &p, cudaStream_t stream);
cudaError_t launch_attn_simt(AttnParams &p, cudaStream_t stream);
cudaError_t launch_merge_n(const MergeNParams &p, cudaStream_t stream);
cudaError_t launch_merge_2(const Merge2Params &p, cudaStream_t stream);

// True when a tensor-core kernel supports these shapes.
bool attn_tc_supported(const AttnParams &p);
bool attn_decode_tc_supported(const AttnParams &p);
// Per-head work items of the tensor-core kernel (pack_g == 0): query rows
// and heads per item -- 128 rows of 2 heads sharing a kv head when Hq / Hkv
// is even, else 256 rows (two 128-row tiles) of 1 head.
struct TcItemShape {
  int rows, heads;
};
TcItemShape attn_tc_item_shape(const AttnParams &p);

// Device status words (one per translation unit that has bounded waits);
// attn_tc_read_status reads (and clears) both tensor-core kernels' words.
unsigned int attn_tc_read_status(bool clear, cudaError_t *err);
unsigned int attn_pair_read_status(bool clear, cudaError_t *err);
unsigned int attn_simt_read_status(bool clear, cudaError_t *err);
unsigned int merge_read_status(bool clear, cudaError_t *err);

}  // namespace cpattn
