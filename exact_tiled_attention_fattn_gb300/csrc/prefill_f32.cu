// fp32 prefill on the CUDA cores: the exact-precision path (tf32 tensor cores
// would not hold fp32-level error). One warp owns one query row and walks the
// visible keys in blocks of 32, one key per lane, folding each block into the
// running (m, l, O) with the online-softmax rule ("The trick: tiles and an
// online softmax", FlashAttention LLM-inference page). O stays unnormalised
// and is divided by l once at the end.
#include "device_common.cuh"
#include "fattn_internal.h"

#include <math_constants.h>

namespace fattn {
namespace {

constexpr int kRowsPerCta = 4;

template <int D>
__global__ void __launch_bounds__(kRowsPerCta * 32) prefill_f32_kernel(const PrefillParams p) {
  __shared__ __align__(16) float sq[kRowsPerCta][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y, b = blockIdx.z;
  const int G = p.Hq / p.Hkv;
  const int hkv = h / G;

  int start, L;
  if (p.cu_seqlens) {
    start = p.cu_seqlens[b];
    const int end = p.cu_seqlens[b + 1];
    if (start < 0 || end < start || end > p.total_rows || end - start > p.N) {
      if (threadIdx.x == 0 && blockIdx.x == 0 && h == 0) record_status(p.status, kStatusDeviceCheck);
      return;
    }
    L = end - start;
  } else {
    start = b * p.N;
    L = p.N;
  }
  const int i = blockIdx.x * kRowsPerCta + warp;
  if (i >= L) return;

  const float* Q = static_cast<const float*>(p.q);
  const float* K = static_cast<const float*>(p.k);
  const float* V = static_cast<const float*>(p.v);
  const size_t qrow = ((size_t)(start + i) * p.Hq + h) * D;
  for (int c = lane; c < D; c += 32) sq[warp][c] = Q[qrow + c];
  __syncwarp();

  const int kend = p.causal ? min(L, i + 1) : L;
  const float sl2 = p.scale * kLog2e;
  const size_t kstride = (size_t)p.Hkv * D;
  const float* Kh = K + ((size_t)start * p.Hkv + hkv) * D;
  const float* Vh = V + ((size_t)start * p.Hkv + hkv) * D;

  float m = -CUDART_INF_F, l = 0.f;
  float o[D / 32];
#pragma unroll
  for (int e = 0; e < D / 32; ++e) o[e] = 0.f;

  for (int j0 = 0; j0 < kend; j0 += 32) {
    const int j = j0 + lane;
    float s = -CUDART_INF_F;
    if (j < kend) {
      const float4* kr = reinterpret_cast<const float4*>(Kh + (size_t)j * kstride);
      float dot = 0.f;
#pragma unroll 8
      for (int c4 = 0; c4 < D / 4; ++c4) {
        const float4 kv = kr[c4];
        dot = fmaf(sq[warp][4 * c4 + 0], kv.x, dot);
        dot = fmaf(sq[warp][4 * c4 + 1], kv.y, dot);
        dot = fmaf(sq[warp][4 * c4 + 2], kv.z, dot);
        dot = fmaf(sq[warp][4 * c4 + 3], kv.w, dot);
      }
      s = dot * sl2;
    }
    float mc = s;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mc = fmaxf(mc, __shfl_xor_sync(0xffffffffu, mc, off));
    const float mn = fmaxf(m, mc);                 // finite: lane 0 always holds a visible key
    const float alpha = exp2f(m - mn);             // e^{m - m'} (0 on the first block)
    const float pj = exp2f(s - mn);                // e^{s_j - m'} (0 for masked lanes)
    float ps = pj;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
    l = l * alpha + ps;
    m = mn;
#pragma unroll
    for (int e = 0; e < D / 32; ++e) o[e] *= alpha;
    const int nk = min(32, kend - j0);
    for (int jj = 0; jj < nk; ++jj) {
      const float w = __shfl_sync(0xffffffffu, pj, jj);
      const float* vr = Vh + (size_t)(j0 + jj) * kstride;
#pragma unroll
      for (int e = 0; e < D / 32; ++e) o[e] = fmaf(w, vr[lane + 32 * e], o[e]);
    }
  }

  float* O = static_cast<float*>(p.o);
  const float inv = 1.f / l;
#pragma unroll
  for (int e = 0; e < D / 32; ++e) O[qrow + lane + 32 * e] = o[e] * inv;
  if (p.lse && lane == 0) {
    const float lse = (m + log2f(l)) * kLn2;
    if (p.cu_seqlens)
      p.lse[(size_t)h * p.total_rows + start + i] = lse;
    else
      p.lse[((size_t)b * p.Hq + h) * p.N + i] = lse;
  }
}

}  // namespace

cudaError_t launch_prefill_f32(const PrefillParams& p, cudaStream_t stream) {
  dim3 grid((p.N + kRowsPerCta - 1) / kRowsPerCta, p.Hq, p.B);
  if (p.d == 128)
    prefill_f32_kernel<128><<<grid, kRowsPerCta * 32, 0, stream>>>(p);
  else
    prefill_f32_kernel<64><<<grid, kRowsPerCta * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace fattn
