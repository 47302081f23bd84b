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
// Mapping: a warp merges whole (batch, row, head) vectors of D values, lanes
// owning D/32 consecutive columns (16-byte fp32 loads at D = 128), so every O
// request is a fully used, coalesced 512-byte line.  Grids cover all rows with
// short CTAs (no grid-stride loop), so uneven per-row work is balanced by the
// scheduler.  fp32 arithmetic, output rounded once.
#include <cuda_bf16.h>
#include <math.h>

#include "cpattn_internal.h"
#include "epilogue.cuh"

namespace cpattn {

// Device status word of the merge kernels (debug-build bounds checks).
__device__ unsigned int g_merge_status;

namespace {

constexpr int kWarps = 8;
constexpr int kRowsInFlight = 4;  // pairwise merge: rows per warp with all their loads in flight

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

// (a) <- merge(a, b), element-wise over rows.  One warp per run of 32
// consecutive rows of one (batch, head): lane l reads the two LSEs of row
// s0 + l (one coalesced 128-byte load per side, contiguous in the [b, h, s]
// layout), computes that row's weights and writes its merged LSE; the rows'
// O vectors (lanes own D/32 consecutive columns) are then merged
// kRowsInFlight at a time with every load issued before any arithmetic, the
// weights broadcast from the row's lane.
template <int D>
__global__ void __launch_bounds__(kWarps * 32) merge2_kernel(const __grid_constant__ Merge2Params p) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const int64_t n_runs = ((int64_t)p.S + 31) / 32;
  const int64_t wid = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (wid >= (int64_t)p.B * p.H * n_runs) return;
  const int64_t s0 = (wid % n_runs) * 32;
  const int h = (int)((wid / n_runs) % p.H);
  const int b = (int)(wid / (n_runs * p.H));
  const int nrow = (int)((int64_t)p.S - s0 < 32 ? (int64_t)p.S - s0 : 32);
  float la = -INFINITY, lb = -INFINITY;
  if (lane < nrow) {
    la = *view_lse(p.a, b, s0 + lane, h);
    lb = *view_lse(p.b, b, s0 + lane, h);
  }
  const MergeW w = merge_weights(la, lb);
#pragma unroll 1
  for (int u0 = 0; u0 < nrow; u0 += kRowsInFlight) {
    float va[kRowsInFlight][E], vb[kRowsInFlight][E];
#pragma unroll
    for (int u = 0; u < kRowsInFlight; ++u) {
      if (u0 + u < nrow) {
        load_row<E>(p.a, b, s0 + u0 + u, h, lane * E, va[u]);
        load_row<E>(p.b, b, s0 + u0 + u, h, lane * E, vb[u]);
      }
    }
#pragma unroll
    for (int u = 0; u < kRowsInFlight; ++u) {
      if (u0 + u < nrow) {  // warp-uniform
        const float wa = __shfl_sync(0xffffffffu, w.wa, u0 + u);
        const float wb = __shfl_sync(0xffffffffu, w.wb, u0 + u);
#pragma unroll
        for (int i = 0; i < E; ++i) va[u][i] = __fmul_rn(wa, va[u][i]) + __fmul_rn(wb, vb[u][i]);
        store_vals<E>(view_row(p.a, b, s0 + u0 + u, h), p.a.f32, lane * E, va[u]);
      }
    }
  }
  if (lane < nrow) *view_lse(p.a, b, s0 + lane, h) = w.lse;
}

// Pass-Q: for item x, rows [0, chunk_rows) of Q chunk x merge slots
// slot0 .. slot0 + count - 1 (ascending KV chunk) into the final output.
// One pass with a running maximum: every group of F partials (their LSE and O
// rows, for R rows at once) is loaded before any of it is used, so each warp
// keeps up to R * F 512-byte rows in
// flight and pays one memory round trip per group.
template <int D, int R, int F>
__global__ void __launch_bounds__(kWarps * 32) mergen_kernel(const __grid_constant__ MergeNParams p) {
  constexpr int E = D / 32;
  constexpr int kInFlight = F;
  const int lane = threadIdx.x & 31;
  const int item = blockIdx.y;
  const int count = p.item_count[item];
  const int slot0 = p.item_slot0[item];
  const int64_t n_rows = (int64_t)p.B * p.chunk_rows * p.H;
  const int64_t r0 = ((int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5)) * R;
  if (r0 >= n_rows) return;
  if (kDebugChecks && count > 0 && (slot0 < 0 || slot0 + count > p.n_part_slots)) {
    if ((threadIdx.x & 31) == 0) atomicOr(&g_merge_status, kStatusBounds);
    return;
  }
  const float *lse0[R];
  const float *o0[R];
  float m[R], sum[R], acc[R][E];
#pragma unroll
  for (int u = 0; u < R; ++u) {
    const int64_t r = r0 + u < n_rows ? r0 + u : r0;  // a duplicate row is computed, not stored
    const int h = (int)(r % p.H);
    const int64_t s = (r / p.H) % p.chunk_rows;
    const int b = (int)(r / ((int64_t)p.H * p.chunk_rows));
    lse0[u] = p.part.lse + (int64_t)slot0 * p.part_lse_stride + (int64_t)b * p.part.lb +
              (int64_t)h * p.part.lh + s;
    o0[u] = reinterpret_cast<const float *>(p.part.o) + (int64_t)slot0 * p.part_o_stride +
            (int64_t)b * p.part.sb + s * p.part.ss + (int64_t)h * p.part.sh + lane * E;
    m[u] = -INFINITY;
    sum[u] = 0.f;
#pragma unroll
    for (int i = 0; i < E; ++i) acc[u][i] = 0.f;
  }
  for (int j0 = 0; j0 < count; j0 += kInFlight) {
    float l[R][kInFlight];
    float v[R][kInFlight][E];
#pragma unroll
    for (int u = 0; u < R; ++u)
#pragma unroll
      for (int x = 0; x < kInFlight; ++x) {
        if (j0 + x < count) {
          l[u][x] = lse0[u][(int64_t)(j0 + x) * p.part_lse_stride];
          load_f32<E>(o0[u] + (int64_t)(j0 + x) * p.part_o_stride, 0, v[u][x]);
        } else {
          l[u][x] = -INFINITY;
#pragma unroll
          for (int i = 0; i < E; ++i) v[u][x][i] = 0.f;
        }
      }
#pragma unroll
    for (int u = 0; u < R; ++u) {
      float mg = l[u][0];
#pragma unroll
      for (int x = 1; x < kInFlight; ++x) mg = fmaxf(mg, l[u][x]);
      const float m_new = fmaxf(m[u], mg);
      if (m_new == -INFINITY) continue;  // nothing visible yet
      const float c = expf(m[u] - m_new);  // 0 when m = -inf
      sum[u] *= c;
#pragma unroll
      for (int i = 0; i < E; ++i) acc[u][i] *= c;
#pragma unroll
      for (int x = 0; x < kInFlight; ++x) {
        const float e = expf(l[u][x] - m_new);  // 0 for padding and empty parts
        sum[u] += e;
#pragma unroll
        for (int i = 0; i < E; ++i) acc[u][i] = fmaf(e, v[u][x][i], acc[u][i]);
      }
      m[u] = m_new;
    }
  }
#pragma unroll
  for (int u = 0; u < R; ++u) {
    const int64_t r = r0 + u;
    if (r >= n_rows) break;
    const int h = (int)(r % p.H);
    const int64_t s = (r / p.H) % p.chunk_rows;
    const int b = (int)(r / ((int64_t)p.H * p.chunk_rows));
    float lse_out = -INFINITY;
    if (m[u] != -INFINITY) {
      const float inv = 1.f / sum[u];
#pragma unroll
      for (int i = 0; i < E; ++i) acc[u][i] *= inv;
      lse_out = m[u] + logf(sum[u]);
    }
    const int64_t abs_row = (int64_t)p.item_row0[item] + s;
    store_vals<E>(view_row(p.out, b, abs_row, h), p.out.f32, lane * E, acc[u]);
    if (lane == 0) *view_lse(p.out, b, abs_row, h) = lse_out;
  }
}

// Few rows, many partials each (decode: a handful of query rows, one
// partial per split-KV piece of every chunk): one CTA per (row, item); warp w
// runs the same online merge over partials w, w + kWarps, w + 2 kWarps, ...,
// and warp 0 then combines the warps' (max, sum, O) states in shared memory.
// Every load round keeps kInFlight partials per warp, kWarps * kInFlight per
// row, in flight.
template <int D>
__global__ void __launch_bounds__(kWarps * 32)
    mergen_split_kernel(const __grid_constant__ MergeNParams p) {
  constexpr int E = D / 32;
  constexpr int kInFlight = 4;
  __shared__ float s_acc[kWarps][D];
  __shared__ float s_m[kWarps], s_sum[kWarps];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int item = blockIdx.y;
  const int count = p.item_count[item];
  const int slot0 = p.item_slot0[item];
  const int64_t r = blockIdx.x;  // the grid has one CTA per row
  if (kDebugChecks && count > 0 && (slot0 < 0 || slot0 + count > p.n_part_slots)) {
    if (threadIdx.x == 0) atomicOr(&g_merge_status, kStatusBounds);
    return;
  }
  const int h = (int)(r % p.H);
  const int64_t s = (r / p.H) % p.chunk_rows;
  const int b = (int)(r / ((int64_t)p.H * p.chunk_rows));
  const float *lse0 = p.part.lse + (int64_t)slot0 * p.part_lse_stride + (int64_t)b * p.part.lb +
                      (int64_t)h * p.part.lh + s;
  const float *o0 = reinterpret_cast<const float *>(p.part.o) + (int64_t)slot0 * p.part_o_stride +
                    (int64_t)b * p.part.sb + s * p.part.ss + (int64_t)h * p.part.sh + lane * E;
  float m = -INFINITY, sum = 0.f, acc[E];
#pragma unroll
  for (int i = 0; i < E; ++i) acc[i] = 0.f;
  for (int j0 = warp; j0 < count; j0 += kWarps * kInFlight) {
    float l[kInFlight], v[kInFlight][E];
#pragma unroll
    for (int x = 0; x < kInFlight; ++x) {
      const int j = j0 + x * kWarps;
      if (j < count) {
        l[x] = lse0[(int64_t)j * p.part_lse_stride];
        load_f32<E>(o0 + (int64_t)j * p.part_o_stride, 0, v[x]);
      } else {
        l[x] = -INFINITY;
#pragma unroll
        for (int i = 0; i < E; ++i) v[x][i] = 0.f;
      }
    }
    float mg = l[0];
#pragma unroll
    for (int x = 1; x < kInFlight; ++x) mg = fmaxf(mg, l[x]);
    const float m_new = fmaxf(m, mg);
    if (m_new == -INFINITY) continue;
    const float c = expf(m - m_new);
    sum *= c;
#pragma unroll
    for (int i = 0; i < E; ++i) acc[i] *= c;
#pragma unroll
    for (int x = 0; x < kInFlight; ++x) {
      const float e = expf(l[x] - m_new);
      sum += e;
#pragma unroll
      for (int i = 0; i < E; ++i) acc[i] = fmaf(e, v[x][i], acc[i]);
    }
    m = m_new;
  }
#pragma unroll
  for (int i = 0; i < E; ++i) s_acc[warp][lane * E + i] = acc[i];
  if (lane == 0) {
    s_m[warp] = m;
    s_sum[warp] = sum;
  }
  __syncthreads();
  if (warp != 0) return;
  float mx = -INFINITY;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) mx = fmaxf(mx, s_m[w]);
  float tot = 0.f, out[E];
#pragma unroll
  for (int i = 0; i < E; ++i) out[i] = 0.f;
  float lse_out = -INFINITY;
  if (mx != -INFINITY) {
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float c = s_m[w] == -INFINITY ? 0.f : expf(s_m[w] - mx);
      tot = fmaf(c, s_sum[w], tot);
#pragma unroll
      for (int i = 0; i < E; ++i) out[i] = fmaf(c, s_acc[w][lane * E + i], out[i]);
    }
    const float inv = 1.f / tot;
#pragma unroll
    for (int i = 0; i < E; ++i) out[i] *= inv;
    lse_out = mx + logf(tot);
  }
  const int64_t abs_row = (int64_t)p.item_row0[item] + s;
  store_vals<E>(view_row(p.out, b, abs_row, h), p.out.f32, lane * E, out);
  if (lane == 0) *view_lse(p.out, b, abs_row, h) = lse_out;
}

}  // namespace

cudaError_t launch_merge_2(const Merge2Params &p, cudaStream_t stream) {
  const int64_t n_warps = (int64_t)p.B * p.H * (((int64_t)p.S + 31) / 32);
  if (n_warps == 0) return cudaSuccess;
  const int64_t grid = (n_warps + kWarps - 1) / kWarps;
  if (p.D == 128) {
    merge2_kernel<128><<<(unsigned)grid, kWarps * 32, 0, stream>>>(p);
  } else if (p.D == 64) {
    merge2_kernel<64><<<(unsigned)grid, kWarps * 32, 0, stream>>>(p);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_merge_n(const MergeNParams &p, cudaStream_t stream) {
  const int64_t n_rows = (int64_t)p.B * p.chunk_rows * p.H;
  if (n_rows == 0 || p.n_items == 0) return cudaSuccess;
  int max_count = 0;
  for (int x = 0; x < p.n_items; ++x) max_count = p.item_count[x] > max_count ? p.item_count[x] : max_count;
  // A row per CTA when rows are few and partials many (the row-per-warp grid
  // would leave most SMs idle and walk each row's partials serially).
  if (n_rows * p.n_items <= 4096 && max_count >= 2 * kWarps) {
    dim3 grid((unsigned)n_rows, p.n_items);
    if (p.D == 128) {
      mergen_split_kernel<128><<<grid, kWarps * 32, 0, stream>>>(p);
    } else if (p.D == 64) {
      mergen_split_kernel<64><<<grid, kWarps * 32, 0, stream>>>(p);
    } else {
      return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
  }
  // Two rows per warp, two partials of each in flight: few registers, so many
  // warps per SM keep the loads in flight.  Measured at the 128K Pass-Q shape
  // (GB/s): 2 x 2 5880, 2 x 4 5620, 1 x 3 5770, 4 x 4 5060, 2 x 8 4220.
  constexpr int kR = 2, kF = 2;
  const int64_t per_cta = (int64_t)kWarps * kR;
  dim3 grid((unsigned)((n_rows + per_cta - 1) / per_cta), p.n_items);
  if (p.D == 128) {
    mergen_kernel<128, kR, kF><<<grid, kWarps * 32, 0, stream>>>(p);
  } else if (p.D == 64) {
    mergen_kernel<64, kR, kF><<<grid, kWarps * 32, 0, stream>>>(p);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

unsigned int merge_read_status(bool clear, cudaError_t *err) {
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_merge_status, sizeof(v));
  if (e == cudaSuccess && clear) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_merge_status, &zero, sizeof(zero));
  }
  if (err) *err = e;
  return v;
}

}  // namespace cpattn
