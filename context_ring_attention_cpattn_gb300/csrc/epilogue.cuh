// Row epilogue shared by the partial-attention kernels: routes one query
// row's normalised partial (O_p, LSE_p) by the pair's role.
//
//   kStore     dst  <- (O_p, LSE_p)                       (final output)
//   kPartial   slot <- (O_p, LSE_p)                       (Pass-Q partial, fp32)
//   kAccInit   acc  <- (O_p, LSE_p)                       (Pass-KV, first step)
//   kAccMerge  acc  <- merge(acc, (O_p, LSE_p))           (Pass-KV, middle steps)
//   kAccFinal  out  <- merge(acc, (O_p, LSE_p))           (Pass-KV, last step)
//
// merge((O_a, L_a), (O_b, L_b)) = (w_a O_a + w_b O_b, L) (products rounded
// separately, so the merge is bitwise symmetric in its two sides) with
// L = log(e^{L_a} + e^{L_b}), w = e^{L_x - L}: the LSE-weighted combination of
// partials over disjoint key sets that lets a CP rank accumulate the full
// attention result as K/V chunks arrive around the ring ("Scaling LLM
// Inference ...", reading notes, section "The communication bottleneck across
// all three axes", CP paragraph; techreport rewrite, section "Context
// Parallelism for Million-Token Contexts", Pass-KV bullet).
#pragma once

#include <cuda_bf16.h>
#include <math.h>

#include "cpattn_internal.h"

namespace cpattn {

struct MergeW {
  float wa, wb, lse;
};

// Weights of the two sides of an LSE merge.  Both empty -> (0, 0, -inf).
__device__ __forceinline__ MergeW merge_weights(float la, float lb) {
  const float m = fmaxf(la, lb);
  if (m == -INFINITY) return {0.f, 0.f, -INFINITY};
  const float ea = expf(la - m);
  const float eb = expf(lb - m);
  const float s = ea + eb;
  const float inv = 1.f / s;
  return {ea * inv, eb * inv, m + logf(s)};
}

template <int N>
__device__ __forceinline__ void store_vals(void *row, int f32, int c0, const float (&v)[N]) {
  if (f32) {
    float *p = reinterpret_cast<float *>(row) + c0;
    if constexpr (N % 4 == 0) {
#pragma unroll
      for (int i = 0; i < N; i += 4)
        *reinterpret_cast<float4 *>(p + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
    } else {
#pragma unroll
      for (int i = 0; i < N; ++i) p[i] = v[i];
    }
  } else {
    __nv_bfloat16 *p = reinterpret_cast<__nv_bfloat16 *>(row) + c0;
    if constexpr (N % 8 == 0) {
#pragma unroll
      for (int i = 0; i < N; i += 8) {
        uint4 w;
        __nv_bfloat162 t0 = __floats2bfloat162_rn(v[i], v[i + 1]);
        __nv_bfloat162 t1 = __floats2bfloat162_rn(v[i + 2], v[i + 3]);
        __nv_bfloat162 t2 = __floats2bfloat162_rn(v[i + 4], v[i + 5]);
        __nv_bfloat162 t3 = __floats2bfloat162_rn(v[i + 6], v[i + 7]);
        w.x = *reinterpret_cast<uint32_t *>(&t0);
        w.y = *reinterpret_cast<uint32_t *>(&t1);
        w.z = *reinterpret_cast<uint32_t *>(&t2);
        w.w = *reinterpret_cast<uint32_t *>(&t3);
        *reinterpret_cast<uint4 *>(p + i) = w;
      }
    } else if constexpr (N % 2 == 0) {
#pragma unroll
      for (int i = 0; i < N; i += 2)
        *reinterpret_cast<__nv_bfloat162 *>(p + i) = __floats2bfloat162_rn(v[i], v[i + 1]);
    } else {
#pragma unroll
      for (int i = 0; i < N; ++i) p[i] = __float2bfloat16_rn(v[i]);
    }
  }
}

template <int N>
__device__ __forceinline__ void load_f32(const float *row, int c0, float (&v)[N]) {
  const float *p = row + c0;
  if constexpr (N % 4 == 0) {
#pragma unroll
    for (int i = 0; i < N; i += 4) {
      float4 t = *reinterpret_cast<const float4 *>(p + i);
      v[i] = t.x; v[i + 1] = t.y; v[i + 2] = t.z; v[i + 3] = t.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < N; ++i) v[i] = p[i];
  }
}

__device__ __forceinline__ void *view_row(const OutView &w, int b, int64_t row, int h) {
  const int64_t off = (int64_t)b * w.sb + row * w.ss + (int64_t)h * w.sh;
  return w.f32 ? (void *)(reinterpret_cast<float *>(w.o) + off)
               : (void *)(reinterpret_cast<__nv_bfloat16 *>(w.o) + off);
}
__device__ __forceinline__ float *view_lse(const OutView &w, int b, int64_t row, int h) {
  return w.lse + (int64_t)b * w.lb + (int64_t)h * w.lh + row;
}

// One query row's destination, resolved once per row.
struct RowSink {
  int mode;
  void *dst;       // row of the destination (out, slot or acc)
  int dst_f32;
  const float *acc;  // accumulator row read by the merge roles
  float wa, wb;    // merge weights (merge roles)

  // The accumulator LSE a merge role combines with (-inf for other roles).
  // When several threads share a row, each reads it before any of them
  // writes the merged LSE in place, and passes it to init().
  __device__ static __forceinline__ float acc_lse(const AttnParams &p, const PairDesc &pd, int b,
                                                  int h, int rel_row) {
    if (pd.mode != kAccMerge && pd.mode != kAccFinal) return -INFINITY;
    return *view_lse(p.acc, b, (int64_t)pd.q_row0 + rel_row, h);
  }

  // rel_row: row inside the pair's q chunk.  lse_p: the partial's LSE.
  // write_lse: this thread writes the LSE (one thread per row and head).
  // acc_lse_old: the accumulator LSE read beforehand (acc_lse), or null to
  // read it here.
  // status: the calling kernel's device status word (debug-build checks).
  __device__ __forceinline__ void init(const AttnParams &p, const PairDesc &pd, int b, int h,
                                       int rel_row, float lse_p, bool write_lse, int slot = -1,
                                       const float *acc_lse_old = nullptr,
                                       unsigned int *status = nullptr) {
    mode = pd.mode;
    if (slot < 0) slot = pd.slot;
    const int64_t abs_row = (int64_t)pd.q_row0 + rel_row;
    if constexpr (kDebugChecks) {
      bool in = b >= 0 && b < p.B && h >= 0 && h < p.Hq;
      if (mode == kPartial)
        in = in && slot >= 0 && slot < p.n_part_slots && rel_row >= 0 && rel_row < p.part_rows;
      else
        in = in && abs_row >= 0 && abs_row < p.q_rows_total;
      if (!in) {
        if (status != nullptr) atomicOr(status, kStatusBounds);
        dst = nullptr;
        acc = nullptr;
        return;
      }
    }
    acc = nullptr;
    wa = 0.f;
    wb = 1.f;
    if (mode == kStore) {
      dst = view_row(p.out, b, abs_row, h);
      dst_f32 = p.out.f32;
      if (write_lse) *view_lse(p.out, b, abs_row, h) = lse_p;
    } else if (mode == kPartial) {
      OutView w = p.part;
      w.o = reinterpret_cast<float *>(w.o) + (int64_t)slot * p.part_o_stride;
      w.lse = w.lse + (int64_t)slot * p.part_lse_stride;
      dst = view_row(w, b, rel_row, h);
      dst_f32 = 1;
      if (write_lse) *view_lse(w, b, rel_row, h) = lse_p;
    } else if (mode == kAccInit) {
      dst = view_row(p.acc, b, abs_row, h);
      dst_f32 = 1;
      if (write_lse) *view_lse(p.acc, b, abs_row, h) = lse_p;
    } else {  // kAccMerge / kAccFinal
      float *acc_lse = view_lse(p.acc, b, abs_row, h);
      acc = reinterpret_cast<const float *>(view_row(p.acc, b, abs_row, h));
      const MergeW mw = merge_weights(acc_lse_old != nullptr ? *acc_lse_old : *acc_lse, lse_p);
      wa = mw.wa;
      wb = mw.wb;
      if (mode == kAccMerge) {
        dst = const_cast<float *>(acc);
        dst_f32 = 1;
        if (write_lse) *acc_lse = mw.lse;
      } else {
        dst = view_row(p.out, b, abs_row, h);
        dst_f32 = p.out.f32;
        if (write_lse) *view_lse(p.out, b, abs_row, h) = mw.lse;
      }
    }
  }

  // Columns [c0, c0 + N) of the row; v holds the normalised partial O_p.
  template <int N>
  __device__ __forceinline__ void put(int c0, float (&v)[N]) const {
    if (kDebugChecks && dst == nullptr) return;  // failed bounds check
    if (acc != nullptr) {
      float a[N];
      load_f32<N>(acc, c0, a);
#pragma unroll
      for (int i = 0; i < N; ++i) v[i] = __fmul_rn(wa, a[i]) + __fmul_rn(wb, v[i]);
    }
    store_vals<N>(dst, dst_f32, c0, v);
  }
};

}  // namespace cpattn
