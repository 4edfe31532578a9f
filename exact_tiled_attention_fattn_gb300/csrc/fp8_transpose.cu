// V transpose for the FP8 prefill: the P V product takes V as its B operand
// with the keys (the reduction dimension) contiguous, so V [B, N, Hkv, d]
// (E4M3 bytes, d contiguous) is rewritten as V^T [B * Hkv, d, Npad] with the
// keys past N zero. One block per (128-key tile, sequence and KV head): the
// tile goes through shared memory so that both the reads (d-long rows) and the
// writes (128-key rows) are 16-byte accesses.
#include "fattn_internal.h"

#include <cuda_runtime.h>
#include <stdint.h>

namespace fattn {
namespace {

constexpr int kKeys = 128;
constexpr int kDim = 128;  // d

__global__ void __launch_bounds__(256) fp8_transpose_v_kernel(const uint8_t* __restrict__ v,
                                                             uint8_t* __restrict__ vt, int N, int Hkv, int Npad) {
  __shared__ uint8_t tile[kKeys][kDim + 16];  // row k: the d bytes of key k (padded)
  const int kb = blockIdx.x, bh = blockIdx.y;
  const int b = bh / Hkv, hkv = bh - b * Hkv;
  for (int id = threadIdx.x; id < kKeys * kDim / 16; id += blockDim.x) {
    const int key = id / (kDim / 16), c16 = id % (kDim / 16);
    const int n = kb * kKeys + key;
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (n < N) val = *reinterpret_cast<const uint4*>(v + (((size_t)b * N + n) * Hkv + hkv) * kDim + c16 * 16);
    *reinterpret_cast<uint4*>(&tile[key][c16 * 16]) = val;
  }
  __syncthreads();
  for (int id = threadIdx.x; id < kDim * kKeys / 16; id += blockDim.x) {
    const int dd = id / (kKeys / 16), k16 = id % (kKeys / 16);
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int k0 = k16 * 16 + 4 * e;
      w[e] = (uint32_t)tile[k0][dd] | ((uint32_t)tile[k0 + 1][dd] << 8) | ((uint32_t)tile[k0 + 2][dd] << 16) |
             ((uint32_t)tile[k0 + 3][dd] << 24);
    }
    *reinterpret_cast<uint4*>(vt + ((size_t)bh * kDim + dd) * Npad + (size_t)kb * kKeys + k16 * 16) =
        make_uint4(w[0], w[1], w[2], w[3]);
  }
}

}  // namespace

cudaError_t launch_fp8_transpose_v(const uint8_t* v, uint8_t* vt, int B, int N, int Hkv, int d, int Npad,
                                   cudaStream_t stream) {
  if (d != kDim || Npad % kKeys) return cudaErrorInvalidValue;
  const dim3 grid(Npad / kKeys, B * Hkv);
  fp8_transpose_v_kernel<<<grid, 256, 0, stream>>>(v, vt, N, Hkv, Npad);
  return cudaGetLastError();
}

}  // namespace fattn
