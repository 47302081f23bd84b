// LSE-weighted merge kernels (memory-bound).
//
// Partials over disjoint key sets combine exactly as
//   LSE = m + log sum_p exp(LSE_p - m),  O = sum_p exp(LSE_p - LSE) O_p,
// the step by which a CP rank turns per-chunk results into attention over the
// full context ("Scaling LLM Inference ...", techreport rewrite, section
// "Context Parallelism for Million-Token Contexts", Pass-Q bullet: query
// tensors visit the ranks, so each Q chunk's partials are combined
// afterwards; reading notes, section "The communication bottleneck across all
// three axes", CP paragraph: ranks accumulate the full attention result).
//
// Mapping: one warp per (batch, row, head) vector of D values, lanes own D/32
// consecutive columns (16-byte fp32 loads at D = 128), consecutive warps walk
// consecutive rows of the [b, s, h, d] layout, so every request is a fully
// used, coalesced 512-byte line.  fp32 arithmetic, output rounded once.
#include <cuda_bf16.h>
#include <math.h>

#include "cpattn_internal.h"
#include "epilogue.cuh"

namespace cpattn {
namespace {

constexpr int kWarps = 8;

template <int E>
__device__ __forceinline__ void load_row(const OutView &w, int b, int64_t row, int h, int c0,
                                         float (&v)[E]) {
  const void *base = view_row(w, b, row, h);
  if (w.f32) {
    load_f32<E>(reinterpret_cast<const float *>(base), c0, v);
  } else {
    const __nv_bfloat16 *p = reinterpret_cast<const __nv_bfloat16 *>(base) + c0;
#pragma unroll
    for (int i = 0; i < E; ++i) v[i] = __bfloat162float(p[i]);
  }
}

// (a) <- merge(a, b), element-wise over rows.
template <int D>
__global__ void __launch_bounds__(kWarps * 32) merge2_kernel(const __grid_constant__ Merge2Params p) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const int64_t n_rows = (int64_t)p.B * p.S * p.H;
  for (int64_t r = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); r < n_rows;
       r += (int64_t)gridDim.x * kWarps) {
    const int h = (int)(r % p.H);
    const int64_t s = (r / p.H) % p.S;
    const int b = (int)(r / ((int64_t)p.H * p.S));
    float *la = view_lse(p.a, b, s, h);
    const float lb = *view_lse(p.b, b, s, h);
    const MergeW w = merge_weights(*la, lb);
    float va[E], vb[E];
    load_row<E>(p.a, b, s, h, lane * E, va);
    load_row<E>(p.b, b, s, h, lane * E, vb);
#pragma unroll
    for (int i = 0; i < E; ++i) va[i] = __fmul_rn(w.wa, va[i]) + __fmul_rn(w.wb, vb[i]);
    __syncwarp();
    store_vals<E>(view_row(p.a, b, s, h), p.a.f32, lane * E, va);
    if (lane == 0) *la = w.lse;
  }
}

// Pass-Q: for item x, rows [0, chunk_rows) of Q chunk x merge slots
// slot0 .. slot0 + count - 1 (ascending KV chunk) into the final output.
// Each warp keeps kInFlight partial rows' loads outstanding at once, so an
// SM has enough bytes in flight to approach the copy bandwidth.
template <int D>
__global__ void __launch_bounds__(kWarps * 32) mergen_kernel(const __grid_constant__ MergeNParams p) {
  constexpr int E = D / 32;
  constexpr int kInFlight = 8;
  const int lane = threadIdx.x & 31;
  const int item = blockIdx.y;
  const int count = p.item_count[item];
  const int slot0 = p.item_slot0[item];
  const int64_t n_rows = (int64_t)p.B * p.chunk_rows * p.H;
  for (int64_t r = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); r < n_rows;
       r += (int64_t)gridDim.x * kWarps) {
    const int h = (int)(r % p.H);
    const int64_t s = (r / p.H) % p.chunk_rows;  // chunk-relative row
    const int b = (int)(r / ((int64_t)p.H * p.chunk_rows));
    const float *lse0 = p.part.lse + (int64_t)slot0 * p.part_lse_stride + (int64_t)b * p.part.lb +
                        (int64_t)h * p.part.lh + s;
    const float *o0 = reinterpret_cast<const float *>(p.part.o) + (int64_t)slot0 * p.part_o_stride +
                      (int64_t)b * p.part.sb + s * p.part.ss + (int64_t)h * p.part.sh + lane * E;
    // Maximum LSE over the parts.
    float m = -INFINITY;
    for (int j0 = 0; j0 < count; j0 += kInFlight) {
#pragma unroll
      for (int u = 0; u < kInFlight; ++u)
        if (j0 + u < count) m = fmaxf(m, lse0[(int64_t)(j0 + u) * p.part_lse_stride]);
    }
    float acc[E];
#pragma unroll
    for (int i = 0; i < E; ++i) acc[i] = 0.f;
    float lse_out = -INFINITY;
    if (m != -INFINITY) {
      float sum = 0.f;
      for (int j0 = 0; j0 < count; j0 += kInFlight) {
        float l[kInFlight];
        float v[kInFlight][E];
#pragma unroll
        for (int u = 0; u < kInFlight; ++u) {
          if (j0 + u < count) {
            l[u] = lse0[(int64_t)(j0 + u) * p.part_lse_stride];
            load_f32<E>(o0 + (int64_t)(j0 + u) * p.part_o_stride, 0, v[u]);
          } else {
            l[u] = -INFINITY;
#pragma unroll
            for (int i = 0; i < E; ++i) v[u][i] = 0.f;
          }
        }
#pragma unroll
        for (int u = 0; u < kInFlight; ++u) {
          const float e = expf(l[u] - m);  // 0 for padding and empty parts
          sum += e;
#pragma unroll
          for (int i = 0; i < E; ++i) acc[i] = fmaf(e, v[u][i], acc[i]);
        }
      }
      const float inv = 1.f / sum;
#pragma unroll
      for (int i = 0; i < E; ++i) acc[i] *= inv;
      lse_out = m + logf(sum);
    }
    const int64_t abs_row = (int64_t)p.item_row0[item] + s;
    store_vals<E>(view_row(p.out, b, abs_row, h), p.out.f32, lane * E, acc);
    if (lane == 0) *view_lse(p.out, b, abs_row, h) = lse_out;
  }
}

int grid_for(int64_t n_rows) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t want = (n_rows + kWarps - 1) / kWarps;
  const int64_t cap = (int64_t)sms * 8;  // 8 resident CTAs of 256 threads per SM
  return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace

cudaError_t launch_merge_2(const Merge2Params &p, cudaStream_t stream) {
  const int64_t n_rows = (int64_t)p.B * p.S * p.H;
  if (n_rows == 0) return cudaSuccess;
  const int grid = grid_for(n_rows);
  if (p.D == 128) {
    merge2_kernel<128><<<grid, kWarps * 32, 0, stream>>>(p);
  } else if (p.D == 64) {
    merge2_kernel<64><<<grid, kWarps * 32, 0, stream>>>(p);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_merge_n(const MergeNParams &p, cudaStream_t stream) {
  const int64_t n_rows = (int64_t)p.B * p.chunk_rows * p.H;
  if (n_rows == 0 || p.n_items == 0) return cudaSuccess;
  int gx = grid_for(n_rows * p.n_items);
  gx = (gx + p.n_items - 1) / p.n_items;
  dim3 grid(gx, p.n_items);
  if (p.D == 128) {
    mergen_kernel<128><<<grid, kWarps * 32, 0, stream>>>(p);
  } else if (p.D == 64) {
    mergen_kernel<64><<<grid, kWarps * 32, 0, stream>>>(p);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace cpattn
