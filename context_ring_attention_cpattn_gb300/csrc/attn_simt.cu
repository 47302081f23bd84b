// Partial attention of (Q-chunk, KV-chunk) pairs on the FP32 pipe (no tensor
// cores).  Serves fp32 inputs -- whose tolerance needs true fp32 products,
// which TF32 tensor-core math would not give -- and head_dim 64 in bf16.
// Same pair/role interface as the tcgen05 kernel.
//
// What one pair computes ("Scaling LLM Inference ...", techreport rewrite,
// section "Context Parallelism for Million-Token Contexts": each rank's
// attention over the chunks it sees): for query row i and head h,
//   s_j = scale * q_i . k_j over keys j with kv_pos(j) <= q_pos(i),
//   LSE = log sum_j exp(s_j), O = sum_j exp(s_j - LSE) v_j,
// evaluated with a running maximum (online softmax) in fp32.
//
// Mapping: a CTA of 8 warps takes 8 consecutive query rows of one head.  K/V
// tiles of 32 rows are staged in shared memory as fp32; lane j of a warp
// scores key j of the tile for the warp's row, then every lane accumulates
// its D/32 output columns.
#include <cuda_bf16.h>
#include <math.h>

#include "cpattn_internal.h"
#include "epilogue.cuh"

namespace cpattn {

// Device status word of this kernel (debug-build bounds checks).
__device__ unsigned int g_attn_simt_status;

namespace {

constexpr int kRows = 8;   // query rows per CTA (one per warp)
constexpr int kTile = 32;  // keys per shared-memory tile

__device__ __forceinline__ float ld_in(const void *base, int64_t off, int f32) {
  return f32 ? reinterpret_cast<const float *>(base)[off]
             : __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(base)[off]);
}

template <int D>
__global__ void __launch_bounds__(kRows * 32) attn_simt_kernel(const __grid_constant__ AttnParams p) {
  constexpr int E = D / 32;  // output columns per lane
  __shared__ float sq[kRows][D];
  __shared__ float sk[kTile][D + 1];
  __shared__ float sv[kTile][D];

  // Decode the work item.
  int pi = 0;
  while (pi + 1 < p.n_pairs && (int)blockIdx.x >= p.pairs[pi + 1].cta_begin) ++pi;
  const PairDesc &pd = p.pairs[pi];
  int local = blockIdx.x - pd.cta_begin;
  const int h = local % p.Hq;
  local /= p.Hq;
  const int b = local % p.B;
  const int qt = pd.n_qtiles - 1 - local / p.B;  // later (longer) rows first
  const int hk = h / (p.Hq / p.Hkv);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i0 = qt * kRows;
  const int rows_here = min(kRows, pd.q_len - i0);
  const int i = i0 + warp;              // this warp's row (relative)
  const bool row_ok = warp < rows_here;

  // Stage the CTA's query rows (fp32).
  for (int x = threadIdx.x; x < kRows * D; x += blockDim.x) {
    const int r = x / D, c = x % D;
    float val = 0.f;
    if (r < rows_here)
      val = ld_in(p.q, (int64_t)b * p.q_sb + (int64_t)(pd.q_row0 + i0 + r) * p.q_ss +
                           (int64_t)h * p.q_sh + c, p.in_f32);
    sq[r][c] = val;
  }

  // Keys this CTA may need: up to the last row's causal limit.
  int64_t kv_end = pd.kv_len;
  if (p.causal) {
    const int64_t lim = (int64_t)(i0 + rows_here - 1) + pd.delta + 1;
    kv_end = lim < kv_end ? lim : kv_end;
  }
  if (kv_end < 0) kv_end = 0;
  // Visible keys of this warp's row: [0, my_end).
  int64_t my_end = pd.kv_len;
  if (p.causal) {
    const int64_t lim = (int64_t)i + pd.delta + 1;
    my_end = lim < my_end ? lim : my_end;
  }
  if (my_end < 0) my_end = 0;

  float m = -INFINITY, l = 0.f;
  float o[E];
#pragma unroll
  for (int e = 0; e < E; ++e) o[e] = 0.f;

  for (int64_t j0 = 0; j0 < kv_end; j0 += kTile) {
    __syncthreads();
    for (int x = threadIdx.x; x < kTile * D; x += blockDim.x) {
      const int r = x / D, c = x % D;
      float kv_k = 0.f, kv_v = 0.f;
      if (j0 + r < kv_end) {
        const int64_t row = pd.kv_row0 + j0 + r;
        kv_k = ld_in(p.k, (int64_t)b * p.k_sb + row * p.k_ss + (int64_t)hk * p.k_sh + c, p.in_f32);
        kv_v = ld_in(p.v, (int64_t)b * p.v_sb + row * p.v_ss + (int64_t)hk * p.v_sh + c, p.in_f32);
      }
      sk[r][c] = kv_k;
      sv[r][c] = kv_v;
    }
    __syncthreads();
    if (!row_ok) continue;
    // Lane j scores key j0 + j.
    float s = 0.f;
#pragma unroll 8
    for (int c = 0; c < D; ++c) s = fmaf(sq[warp][c], sk[lane][c], s);
    s *= p.scale;
    const bool vis = (j0 + lane) < my_end;
    if (!vis) s = -INFINITY;
    float tmax = s;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
    const float m_new = fmaxf(m, tmax);
    if (m_new == -INFINITY) continue;  // nothing visible yet for this row
    const float corr = expf(m - m_new);  // m = -inf -> 0
    const float pj = vis ? expf(s - m_new) : 0.f;
    float psum = pj;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
    l = l * corr + psum;
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] *= corr;
#pragma unroll 4
    for (int j = 0; j < kTile; ++j) {
      const float w = __shfl_sync(0xffffffffu, pj, j);
#pragma unroll
      for (int e = 0; e < E; ++e) o[e] = fmaf(w, sv[j][lane * E + e], o[e]);
    }
    m = m_new;
  }

  if (!row_ok) return;
  const float inv = l > 0.f ? 1.f / l : 0.f;
  const float lse = l > 0.f ? m + logf(l) : -INFINITY;
#pragma unroll
  for (int e = 0; e < E; ++e) o[e] *= inv;
  RowSink sink;
  sink.init(p, pd, b, h, i, lse, lane == 0, -1, nullptr, &g_attn_simt_status);
  sink.put<E>(lane * E, o);
}

}  // namespace

cudaError_t launch_attn_simt(AttnParams &p, cudaStream_t stream) {
  int total = 0;
  for (int x = 0; x < p.n_pairs; ++x) {
    PairDesc &pd = p.pairs[x];
    pd.n_qtiles = (pd.q_len + kRows - 1) / kRows;
    pd.cta_begin = total;
    total += pd.n_qtiles * p.Hq * p.B;
  }
  p.total_ctas = total;
  if (total == 0) return cudaSuccess;
  dim3 grid(total), block(kRows * 32);
  if (p.D == 64) {
    attn_simt_kernel<64><<<grid, block, 0, stream>>>(p);
  } else if (p.D == 128) {
    attn_simt_kernel<128><<<grid, block, 0, stream>>>(p);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

unsigned int attn_simt_read_status(bool clear, cudaError_t *err) {
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_attn_simt_status, sizeof(v));
  if (e == cudaSuccess && clear) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_attn_simt_status, &zero, sizeof(zero));
  }
  if (err) *err = e;
  return v;
}

}  // namespace cpattn
