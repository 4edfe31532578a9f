// V transpose for the FP8 prefill: the P V product takes V as its B operand
// with the keys (the reduction dimension) contiguous, so V [B, N, Hkv, d]
// (E4M3 bytes, d contiguous) is rewritten as V^T [B * Hkv, d, Npad] with the
// keys past N zero. One block of 128 threads per (128-key tile, sequence and
// KV head): the tile is read with 16-byte loads into shared memory (rows of
// 144 bytes, so that both phases are free of bank conflicts); then each thread
// takes 4 bytes of d from each of 32 keys (one 32-bit read per key), turns the
// 32 x 4 byte block around with byte permutes, and writes 32 keys of each of
// its 4 rows of V^T as whole 32-byte sectors.
#include "fattn_internal.h"

#include <cuda_runtime.h>
#include <stdint.h>

namespace fattn {
namespace {

constexpr int kKeys = 128;
constexpr int kDim = 128;              // d
constexpr int kRowWords = kDim / 4 + 4;  // 144-byte rows

__global__ void __launch_bounds__(128) fp8_transpose_v_kernel(const uint8_t* __restrict__ v,
                                                             uint8_t* __restrict__ vt, int N, int Hkv, int Npad) {
  __shared__ __align__(16) uint32_t tile[kKeys * kRowWords];  // row k: the d bytes of key k
  const int kb = blockIdx.x, bh = blockIdx.y;
  const int b = bh / Hkv, hkv = bh - b * Hkv;
#pragma unroll
  for (int i = 0; i < kKeys * kDim / 16 / 128; ++i) {
    const int id = i * 128 + threadIdx.x;
    const int key = id / (kDim / 16), c16 = id % (kDim / 16);
    const int n = kb * kKeys + key;
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (n < N) val = *reinterpret_cast<const uint4*>(v + (((size_t)b * N + n) * Hkv + hkv) * kDim + c16 * 16);
    *reinterpret_cast<uint4*>(&tile[key * kRowWords + 4 * c16]) = val;
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;  // d bytes 4 lane .. 4 lane + 3; keys 32 w .. 32 w + 31
  uint32_t u[32];
#pragma unroll
  for (int kk = 0; kk < 32; ++kk) u[kk] = tile[(32 * w + kk) * kRowWords + lane];
#pragma unroll
  for (int dd = 0; dd < 4; ++dd) {
    const uint32_t sel = (uint32_t)dd | ((uint32_t)(dd + 4) << 4);  // byte dd of x, then byte dd of y
    uint32_t o[8];
#pragma unroll
    for (int g = 0; g < 8; ++g) {  // keys 4 g .. 4 g + 3
      const uint32_t lo = __byte_perm(u[4 * g], u[4 * g + 1], sel);
      const uint32_t hi = __byte_perm(u[4 * g + 2], u[4 * g + 3], sel);
      o[g] = __byte_perm(lo, hi, 0x5410);
    }
    uint4* dst = reinterpret_cast<uint4*>(vt + ((size_t)bh * kDim + 4 * lane + dd) * Npad + (size_t)kb * kKeys + 32 * w);
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

}  // namespace

cudaError_t launch_fp8_transpose_v(const uint8_t* v, uint8_t* vt, int B, int N, int Hkv, int d, int Npad,
                                   cudaStream_t stream) {
  if (d != kDim || Npad % kKeys) return cudaErrorInvalidValue;
  const dim3 grid(Npad / kKeys, B * Hkv);
  fp8_transpose_v_kernel<<<grid, 128, 0, stream>>>(v, vt, N, Hkv, Npad);
  return cudaGetLastError();
}

}  // namespace fattn
