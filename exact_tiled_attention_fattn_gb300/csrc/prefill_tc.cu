// Tensor-core prefill for sm_103a: exact attention tile by tile with the
// online-softmax rule ("The trick: tiles and an online softmax", FlashAttention
// LLM-inference page; "The forward pass", FlashAttention explained).
//
// One CTA per SM loops over work items (sequence, query head, 128-row Q tile).
// Roles (warp-specialised):
//   warp 0      TMA producer: Q tile once per item, then K_j / V_j tiles into
//               two 2-stage rings (128-byte swizzle, 64-column boxes).
//   warp 1      MMA issuer (one thread): S_j = Q K_j^T into one of two TMEM
//               score buffers, O += P_j V_j with P_j read from TMEM.
//   warps 2-5   softmax: each thread owns one query row (TMEM lane). It loads
//               its 128 scores, masks (causal diagonal, sequence end), keeps
//               the running max m and sum l in registers, writes P_j (bf16) to
//               TMEM, rescales O in TMEM by e^{m-m'} when the max moved, and
//               at the end writes O / l (bf16) and lse = m + ln l.
// Causal tiles above the diagonal are never loaded or computed ("tiles above
// the diagonal are never touched"). S and P never leave the SM.
//
// Every pipeline wait is bounded: a wait that exceeds its limit records
// FATTN_ERR_TIMEOUT in the device status word, every role stops, in-flight
// copies and MMAs are drained, TMEM is freed and the kernel returns.
#include "device_common.cuh"
#include "fattn_internal.h"
#include "sm100_primitives.cuh"

#include <math_constants.h>

namespace fattn {
namespace {

using namespace sm100;

constexpr int BM = 128;          // query rows per tile (M of one tcgen05.mma)
constexpr int BN = 128;          // keys per tile
constexpr int kThreads = 192;    // 6 warps
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait
constexpr uint64_t kDrainLimitNs = 200000000ull;  // 0.2 s per drain wait

template <int D>
struct TcLayout {
  static constexpr int kQBytes = BM * D * 2;
  static constexpr int kKVBytes = BN * D * 2;
  static constexpr int kStages = 2;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQBytes;
  static constexpr int kOffV = kOffK + kStages * kKVBytes;
  static constexpr int kOffBar = kOffV + kStages * kKVBytes;
  static constexpr int kNumBars = 16;
  static constexpr int kOffHolder = kOffBar + kNumBars * 8;
  static constexpr int kOffAbort = kOffHolder + 8;
  // + slack to align the base to 1024 B; at least 117 KB so that a second CTA
  // (which would block in tcgen05.alloc) never shares the SM
  static constexpr int kUsed = kOffAbort + 8 + 1024;
  static constexpr int kBytes = kUsed > 117 * 1024 ? kUsed : 117 * 1024;
  // TMEM columns: two fp32 score buffers, the fp32 output, two bf16 P buffers.
  static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256;
  static constexpr uint32_t kColP0 = 256 + D, kColP1 = 256 + D + BN / 2;
  static_assert(kColP1 + BN / 2 <= kTmemCols, "TMEM budget");
};

// barrier slots
enum : int {
  kBarQFull = 0, kBarQEmpty = 1, kBarKFull = 2, kBarKEmpty = 4, kBarVFull = 6, kBarVEmpty = 8,
  kBarSFull = 10, kBarPFull = 12, kBarOFull = 14, kBarMmaDone = 15
};

struct Item {
  int b, h, mt, row0, L, n;
  bool valid;
};

__device__ __forceinline__ Item decode_item(const PrefillParams& p, int it, int tiles) {
  Item x;
  const int bh = it / tiles;
  x.mt = tiles - 1 - (it - bh * tiles);  // heaviest Q tile of a head first
  x.b = bh / p.Hq;
  x.h = bh - x.b * p.Hq;
  if (p.cu_seqlens) {
    const int start = __ldg(p.cu_seqlens + x.b);
    const int end = __ldg(p.cu_seqlens + x.b + 1);
    if (start < 0 || end < start || end > p.total_rows || end - start > p.N) {
      x.valid = false;
      x.row0 = x.L = x.n = 0;
      if (x.mt == 0 && x.h == 0 && (threadIdx.x & 31) == 0) record_status(p.status, kStatusDeviceCheck);
      return x;
    }
    x.row0 = start;
    x.L = end - start;
  } else {
    x.row0 = x.b * p.N;
    x.L = p.N;
  }
  x.valid = x.mt * BM < x.L;
  const int kv_tiles = (x.L + BN - 1) / BN;
  x.n = p.causal ? min(x.mt + 1, kv_tiles) : kv_tiles;
  return x;
}

// Drain wait: bounded, ignores the abort flag (used on the way out).
__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kDrainLimitNs) break;
  }
}

// Warp-uniform wait: lane 0 polls, the verdict is broadcast so that every
// lane takes the same path into the warp-collective tcgen05.ld/st.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort, int* status) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort, status, kWaitLimitNs);
  ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  return ok;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                      const __grid_constant__ CUtensorMap tv, const PrefillParams p) {
  using Lay = TcLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sb + Lay::kOffBar + 8 * i; };
  volatile int* abort = reinterpret_cast<volatile int*>(smem + Lay::kOffAbort);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < Lay::kNumBars; ++i) mbar_init(bar(i), (i == kBarPFull || i == kBarPFull + 1) ? 4 : 1);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tq);
    tma_prefetch_desc(&tk);
    tma_prefetch_desc(&tv);
  }
  if (warp == 1) {
    tmem_alloc(sb + Lay::kOffHolder, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + Lay::kOffHolder);

  const int tiles = (p.N + BM - 1) / BM;
  const int num_items = p.B * p.Hq * tiles;
  const int G = p.Hq / p.Hkv;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t nq = 0, nk = 0, nv = 0;
      const uint64_t pol_q = policy_evict_first(), pol_kv = policy_evict_last();
      for (int it = blockIdx.x; it < num_items; it += gridDim.x) {
        const Item x = decode_item(p, it, tiles);
        if (!x.valid) continue;
        const int hkv = x.h / G;
        if (!mbar_wait(bar(kBarQEmpty), (nq & 1) ^ 1, abort, p.status, kWaitLimitNs)) break;
        mbar_arrive_expect_tx(bar(kBarQFull), Lay::kQBytes);
#pragma unroll
        for (int dc = 0; dc < D / 64; ++dc)
          tma_load_3d(sb + Lay::kOffQ + dc * BM * 128, &tq, bar(kBarQFull), dc * 64, x.h, x.row0 + x.mt * BM, pol_q);
        ++nq;
        auto load_k = [&](int j) -> bool {
          const uint32_t st = nk & 1;
          if (!mbar_wait(bar(kBarKEmpty + st), ((nk >> 1) & 1) ^ 1, abort, p.status, kWaitLimitNs)) return false;
          mbar_arrive_expect_tx(bar(kBarKFull + st), Lay::kKVBytes);
#pragma unroll
          for (int dc = 0; dc < D / 64; ++dc)
            tma_load_3d(sb + Lay::kOffK + st * Lay::kKVBytes + dc * BN * 128, &tk, bar(kBarKFull + st), dc * 64,
                        hkv, x.row0 + j * BN, pol_kv);
          ++nk;
          return true;
        };
        auto load_v = [&](int j) -> bool {
          const uint32_t st = nv & 1;
          if (!mbar_wait(bar(kBarVEmpty + st), ((nv >> 1) & 1) ^ 1, abort, p.status, kWaitLimitNs)) return false;
          mbar_arrive_expect_tx(bar(kBarVFull + st), Lay::kKVBytes);
#pragma unroll
          for (int dc = 0; dc < D / 64; ++dc)
            tma_load_3d(sb + Lay::kOffV + st * Lay::kKVBytes + dc * BN * 128, &tv, bar(kBarVFull + st), dc * 64,
                        hkv, x.row0 + j * BN, pol_kv);
          ++nv;
          return true;
        };
        // same order the MMA warp consumes them: K0 K1 V0 K2 V1 K3 V2 ...
        bool ok = load_k(0) && (x.n < 2 || load_k(1)) && load_v(0);
        for (int j = 2; ok && j < x.n; ++j) ok = load_k(j) && load_v(j - 1);
        if (ok && x.n > 1) ok = load_v(x.n - 1);
        if (!ok) break;
      }
      // no copy may land after the CTA is gone: wait for the last armed phase of each barrier
      if (nq) mbar_drain(bar(kBarQFull), (nq - 1) & 1);
      for (uint32_t st = 0; st < 2; ++st) {
        const uint32_t ck = (nk + 1 - st) / 2, cv = (nv + 1 - st) / 2;  // loads issued into stage st
        if (ck) mbar_drain(bar(kBarKFull + st), (ck - 1) & 1);
        if (cv) mbar_drain(bar(kBarVFull + st), (cv - 1) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(BM, BN, 0);  // Q K^T: both K-major
      constexpr uint32_t idO = idesc_bf16_f32(BM, D, 1);   // P V: V is MN-major (d contiguous)
      uint32_t nq = 0, nk = 0, nv = 0, gs = 0;
      bool ok = true;
      for (int it = blockIdx.x; ok && it < num_items; it += gridDim.x) {
        const Item x = decode_item(p, it, tiles);
        if (!x.valid) continue;
        if (!mbar_wait(bar(kBarQFull), nq & 1, abort, p.status, kWaitLimitNs)) break;
        ++nq;
        tc_fence_after();
        auto issue_s = [&](uint32_t g) -> bool {
          const uint32_t st = nk & 1;
          if (!mbar_wait(bar(kBarKFull + st), (nk >> 1) & 1, abort, p.status, kWaitLimitNs)) return false;
          tc_fence_after();
          const uint32_t d_tmem = tmem + ((g & 1) ? Lay::kColS1 : Lay::kColS0);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t a = sb + Lay::kOffQ + (ks >> 2) * BM * 128 + (ks & 3) * 32;
            const uint32_t b = sb + Lay::kOffK + st * Lay::kKVBytes + (ks >> 2) * BN * 128 + (ks & 3) * 32;
            mma_ss(d_tmem, smem_desc_sw128(a, 16, 1024), smem_desc_sw128(b, 16, 1024), idS, ks > 0 ? 1u : 0u);
          }
          mma_commit(bar(kBarKEmpty + st));
          mma_commit(bar(kBarSFull + (g & 1)));
          ++nk;
          return true;
        };
        ok = issue_s(gs) && (x.n < 2 || issue_s(gs + 1));
        if (ok && x.n <= 2) mma_commit(bar(kBarQEmpty));
        for (int j = 0; ok && j < x.n; ++j) {
          const uint32_t g = gs + j;
          if (!mbar_wait(bar(kBarPFull + (g & 1)), (g >> 1) & 1, abort, p.status, kWaitLimitNs)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = nv & 1;
          if (!mbar_wait(bar(kBarVFull + st), (nv >> 1) & 1, abort, p.status, kWaitLimitNs)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t p_tmem = tmem + ((g & 1) ? Lay::kColP1 : Lay::kColP0);
#pragma unroll
          for (int ks = 0; ks < BN / 16; ++ks) {
            const uint32_t b = sb + Lay::kOffV + st * Lay::kKVBytes + ks * 16 * 128;
            mma_ts(tmem + Lay::kColO, p_tmem + ks * 8, smem_desc_sw128(b, BN * 128, 1024), idO,
                   (j > 0 || ks > 0) ? 1u : 0u);
          }
          mma_commit(bar(kBarVEmpty + st));
          mma_commit(bar(kBarOFull));
          ++nv;
          if (j + 2 < x.n) {
            if (!issue_s(g + 2)) {
              ok = false;
              break;
            }
            if (j + 2 == x.n - 1) mma_commit(bar(kBarQEmpty));
          }
        }
        gs += x.n;
      }
      // every MMA (and every commit before this one) has landed before TMEM is freed
      mma_commit(bar(kBarMmaDone));
      mbar_drain(bar(kBarMmaDone), 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int q4 = warp & 3;                 // TMEM lane quarter this warp may touch
    const int r = q4 * 32 + lane;            // query row within the tile
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const float sl2 = p.scale * kLog2e;      // scores go to the log2 domain
    const bool neg = sl2 < 0.f;
    uint32_t gs = 0;
    bool ok = true;
    for (int it = blockIdx.x; ok && it < num_items; it += gridDim.x) {
      const Item x = decode_item(p, it, tiles);
      if (!x.valid) continue;
      const int row = x.mt * BM + r;
      const int lim = p.causal ? min(row + 1, x.L) : x.L;  // keys < lim are visible
      float m = -CUDART_INF_F, l = 0.f;
      for (int j = 0; j < x.n; ++j) {
        const uint32_t g = gs + j;
        if (!warp_wait(bar(kBarSFull + (g & 1)), (g >> 1) & 1, abort, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t s_col = tmem + lane_off + ((g & 1) ? Lay::kColS1 : Lay::kColS0);
        float s[BN];
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t u[32];
          tmem_ld32(s_col + 32 * c, u);
#pragma unroll
          for (int e = 0; e < 32; ++e) s[32 * c + e] = __uint_as_float(u[e]);
        }
        const int kbase = j * BN;
        const bool masked = kbase + BN > lim;  // causal diagonal tile or sequence end
        if (masked) {
#pragma unroll
          for (int c = 0; c < BN; ++c)
            if (kbase + c >= lim) s[c] = neg ? CUDART_INF_F : -CUDART_INF_F;
        }
        float mx = s[0];
        if (!neg) {
#pragma unroll
          for (int c = 1; c < BN; ++c) mx = fmaxf(mx, s[c]);
        } else {
#pragma unroll
          for (int c = 1; c < BN; ++c) mx = fminf(mx, s[c]);
        }
        const float m_new = fmaxf(m, mx * sl2);
        const float base = m_new == -CUDART_INF_F ? 0.f : m_new;
        const float alpha = ex2(m - base);  // e^{m - m'}
        float sum = 0.f;
        uint32_t pk[BN / 2];
        if (!masked) {
#pragma unroll
          for (int c = 0; c < BN; c += 2) {
            const float p0 = ex2(fmaf(s[c], sl2, -base));
            const float p1 = ex2(fmaf(s[c + 1], sl2, -base));
            sum += p0 + p1;
            pk[c / 2] = pack_bf16x2(p0, p1);
          }
        } else {
          const int vis = lim - kbase;  // keys [0, vis) of this tile are visible
#pragma unroll
          for (int c = 0; c < BN; c += 2) {
            const float p0 = c < vis ? ex2(fmaf(s[c], sl2, -base)) : 0.f;
            const float p1 = c + 1 < vis ? ex2(fmaf(s[c + 1], sl2, -base)) : 0.f;
            sum += p0 + p1;
            pk[c / 2] = pack_bf16x2(p0, p1);
          }
        }
        l = l * alpha + sum;
        m = m_new;
        if (j > 0) {
          // PV_{g-1} has landed: O may be rescaled, and P buffer g&1 (read by PV_{g-2}) is free.
          if (!warp_wait(bar(kBarOFull), (g - 1) & 1, abort, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              uint32_t u[32];
              tmem_ld32(tmem + lane_off + Lay::kColO + 32 * c, u);
#pragma unroll
              for (int e = 0; e < 32; ++e) u[e] = __float_as_uint(__uint_as_float(u[e]) * alpha);
              tmem_st32(tmem + lane_off + Lay::kColO + 32 * c, u);
            }
          }
        }
        const uint32_t p_col = tmem + lane_off + ((g & 1) ? Lay::kColP1 : Lay::kColP0);
#pragma unroll
        for (int c = 0; c < BN / 64; ++c) {
          uint32_t u[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) u[e] = pk[32 * c + e];
          tmem_st32(p_col + 32 * c, u);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarPFull + (g & 1)));
      }
      if (!ok) break;
      // epilogue: O / l in bf16 and the row's logsumexp
      if (!warp_wait(bar(kBarOFull), (gs + x.n - 1) & 1, abort, p.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool live = row < x.L;
      const float inv = 1.f / l;
      __nv_bfloat16* orow =
          static_cast<__nv_bfloat16*>(p.o) + ((size_t)(x.row0 + row) * p.Hq + x.h) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t u[32];
        tmem_ld32(tmem + lane_off + Lay::kColO + 32 * c, u);
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          w[e] = pack_bf16x2(__uint_as_float(u[2 * e]) * inv, __uint_as_float(u[2 * e + 1]) * inv);
        if (live) {
          uint4* dst = reinterpret_cast<uint4*>(orow + 32 * c);
#pragma unroll
          for (int e = 0; e < 4; ++e) dst[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
        }
      }
      if (live && p.lse) {
        const float lse = (m + log2f(l)) * kLn2;
        if (p.cu_seqlens)
          p.lse[(size_t)x.h * p.total_rows + x.row0 + row] = lse;
        else
          p.lse[((size_t)x.b * p.Hq + x.h) * p.N + row] = lse;
      }
      gs += x.n;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D>
cudaError_t launch_t(const PrefillParams& p, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                     int num_sms, cudaStream_t stream) {
  using Lay = TcLayout<D>;
  auto kern = prefill_tc_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kBytes);
  if (e != cudaSuccess) return e;
  const long long tiles = (p.N + BM - 1) / BM;
  const long long items = (long long)p.B * p.Hq * tiles;
  if (items > 0x7fffffffLL) return cudaErrorInvalidValue;
  const int grid = (int)(items < num_sms ? items : num_sms);
  kern<<<grid, kThreads, Lay::kBytes, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_tc(const PrefillParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                              const CUtensorMap& tv, int num_sms, cudaStream_t stream) {
  if (p.d == 128) return launch_t<128>(p, tq, tk, tv, num_sms, stream);
  return launch_t<64>(p, tq, tk, tv, num_sms, stream);
}

}  // namespace fattn
