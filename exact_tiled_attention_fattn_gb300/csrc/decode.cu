// Split-KV paged decode ("Flash-Decoding" and "Paged variants" on the
// FlashAttention LLM-inference page) and the merge of split partials with the
// online-softmax rule.
//
// Decode is bound by HBM bandwidth: one query row per (sequence, head) meets a
// long K/V. A persistent grid takes work items (sequence, KV head, split) from
// a counter in the workspace, highest split first; an item covers all query
// heads of that KV head's GQA group (up to 16), so each K/V byte is read once,
// and an empty split costs one atomic instead of a thread block. Each of the
// 4 warps streams its own 16-token chunks through a 2-stage cp.async pipeline
// (16-byte copies, L1 bypassed; two CTAs per SM at d = 128, set by registers), finds each token's page
// through the block table, and runs the two small products on the tensor
// cores with mma.sync (S = Q K^T with the group's heads as the 16 rows,
// O += P V with P kept in registers). Each warp keeps its own running (m, l, O)
// and the four states are merged in shared memory with the same rescaling
// rule at the end. The CTA that finishes the last non-empty split of a
// (sequence, KV-head group) merges that group's partials into the output
// ("Flash-Decoding": partials merged with the same online-softmax rule), so no
// separate merge launch is needed.
#include "device_common.cuh"
#include "fattn_internal.h"

#include <math_constants.h>

namespace fattn {
namespace {

constexpr int kChunk = 16;   // tokens per warp per pipeline stage
constexpr int kWarps = 4;
constexpr int kStages = 2;

template <int D>
struct DecodeLayout {
  static constexpr int kUnits = D / 8;                       // 16-byte units per row
  static constexpr int kStageUnits = 2 * kChunk * kUnits;    // K then V
  static constexpr int kKvUnits = kWarps * kStages * kStageUnits;
  static constexpr int kQUnits = 16 * kUnits;
  static constexpr size_t kBytes = size_t(kKvUnits + kQUnits) * 16;
  // merge scratch (aliases the K/V stages after the main loop)
  static constexpr size_t kMergeBytes = size_t(kWarps) * 16 * (D + 2) * 4;
  static_assert(kMergeBytes <= size_t(kKvUnits) * 16, "merge scratch must fit in the stage buffers");
};

// Row-major rows of D bf16 split into 16-byte units; unit u of row r is stored
// at position u ^ (r & 7) so that 8 consecutive rows read by ldmatrix hit 8
// different bank groups.
template <int D>
__device__ __forceinline__ int swz(int row, int unit) {
  return row * (D / 8) + (unit ^ (row & 7));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D(16x8, f32) += A(16x16, bf16, row) * B(16x8, bf16, col)
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Partial (lse_s, O_s / l_s) of one non-empty split [t0, t1) of sequence b
// for the query heads h0 .. h0 + rows_valid - 1 of KV head hkv.
template <int D, bool kPage16>
__device__ __forceinline__ void decode_split(const DecodeParams& p, uint8_t* smem, int split, int b, int hkv, int h0,
                                             int rows_valid, int t0, int t1) {
  using Lay = DecodeLayout<D>;
  constexpr int U = D / 8;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t q_base = sbase + Lay::kKvUnits * 16;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t prow0 = ((size_t)b * p.Hq + h0) * p.num_splits + split;  // partial row of head h0
  const int nchunks = (t1 - t0 + kChunk - 1) / kChunk;

  // ---- Q rows of the group (rows past the group are zero) ----
  const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(p.q);
  for (int idx = threadIdx.x; idx < 16 * U; idx += kWarps * 32) {
    const int r = idx / U, u = idx % U;
    uint4 val = make_uint4(0, 0, 0, 0);
    if (r < rows_valid) val = *reinterpret_cast<const uint4*>(qg + ((size_t)b * p.Hq + h0 + r) * D + u * 8);
    *reinterpret_cast<uint4*>(smem + Lay::kKvUnits * 16 + swz<D>(r, u) * 16) = val;
  }
  __syncthreads();

  // A fragments of Q for every 16-wide slice of d
  uint32_t qa[D / 16][4];
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const int r = (lane & 7) + ((lane >> 3) & 1) * 8;
    const int u = kk * 2 + (lane >> 4);
    ldsm_x4(q_base + swz<D>(r, u) * 16, qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
  }

  const __nv_bfloat16* kc = static_cast<const __nv_bfloat16*>(p.kcache);
  const __nv_bfloat16* vc = static_cast<const __nv_bfloat16*>(p.vcache);
  const int32_t* table = p.block_table + (size_t)b * p.max_pages_per_seq;
  const uint32_t wbase = sbase + warp * kStages * Lay::kStageUnits * 16;

  // Issue the copies of chunk c into stage st; returns the bit mask of tokens
  // that exist and sit on a valid page.
  auto load_chunk = [&](int c, int st) -> uint32_t {
    const int tb = t0 + c * kChunk;
    const int r = lane & 15;
    const int t = tb + r;
    int page = 0;
    bool ok = false;
    if (lane < 16 && t < t1) {
      const int pi = kPage16 ? (t >> 4) : t / p.page_size;
      page = table[pi];
      ok = (unsigned)page < (unsigned)p.num_pages;
      if (!ok) record_status(p.status, kStatusDeviceCheck);
    }
    const uint32_t vmask = __ballot_sync(0xffffffffu, ok);
    const uint32_t kdst = wbase + st * Lay::kStageUnits * 16;
    const uint32_t vdst = kdst + kChunk * U * 16;
#pragma unroll
    for (int i = 0; i < kChunk * U / 32; ++i) {
      const int idx = lane + 32 * i;
      const int rr = idx / U, u = idx % U;
      const int pg = __shfl_sync(0xffffffffu, page, rr);
      const bool okr = (vmask >> rr) & 1u;
      const int tt = tb + rr;
      const int slot = kPage16 ? (tt & 15) : (tt % p.page_size);
      const size_t off = okr ? ((((size_t)pg * p.page_size + slot) * p.Hkv + hkv) * D + u * 8) : 0;
      const int nbytes = okr ? 16 : 0;
      cp_async16(kdst + swz<D>(rr, u) * 16, kc + off, nbytes);
      cp_async16(vdst + swz<D>(rr, u) * 16, vc + off, nbytes);
    }
    return vmask;
  };

  const float sl2 = p.scale * kLog2e;
  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F;  // rows g and g+8 (log2 domain)
  float l0 = 0.f, l1 = 0.f;                      // this lane's share of the row sums

  const int n_mine = warp < nchunks ? (nchunks - warp + kWarps - 1) / kWarps : 0;
  uint32_t masks[kStages];
#pragma unroll
  for (int i = 0; i < kStages - 1; ++i) {
    masks[i] = i < n_mine ? load_chunk(warp + i * kWarps, i) : 0u;
    cp_async_commit();
  }

  for (int i = 0; i < n_mine; ++i) {
    const int nxt = i + kStages - 1;
    const int st = i % kStages;
    if (nxt < n_mine) masks[nxt % kStages] = load_chunk(warp + nxt * kWarps, nxt % kStages);
    cp_async_commit();
    cp_async_wait<kStages - 1>();
    __syncwarp();
    const uint32_t vm = masks[st];
    const uint32_t kb = wbase + st * Lay::kStageUnits * 16;
    const uint32_t vb = kb + kChunk * U * 16;

    // S = Q K^T for 16 tokens (two 8-token column tiles)
    float s[2][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) s[0][j] = s[1][j] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const int r = (lane & 7) + (lane >> 4) * 8;
      const int u = kk * 2 + ((lane >> 3) & 1);
      uint32_t b0, b1, b2, b3;
      ldsm_x4(kb + swz<D>(r, u) * 16, b0, b1, b2, b3);
      mma_bf16(s[0], qa[kk], b0, b1);
      mma_bf16(s[1], qa[kk], b2, b3);
    }
    // scale into the log2 domain, mask missing tokens, running max per row
    float mx0 = -CUDART_INF_F, mx1 = -CUDART_INF_F;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int tok = nt * 8 + 2 * (lane & 3) + (j & 1);
        const bool ok = (vm >> tok) & 1u;
        s[nt][j] = ok ? s[nt][j] * sl2 : -CUDART_INF_F;
      }
      mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
      mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float base0 = mn0 == -CUDART_INF_F ? 0.f : mn0;
    const float base1 = mn1 == -CUDART_INF_F ? 0.f : mn1;
    const float a0 = ex2(m0 - base0), a1 = ex2(m1 - base1);  // e^{m - m'}
    m0 = mn0;
    m1 = mn1;
    float ps[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      ps[nt][0] = ex2(s[nt][0] - base0);
      ps[nt][1] = ex2(s[nt][1] - base0);
      ps[nt][2] = ex2(s[nt][2] - base1);
      ps[nt][3] = ex2(s[nt][3] - base1);
    }
    l0 = l0 * a0 + ps[0][0] + ps[0][1] + ps[1][0] + ps[1][1];
    l1 = l1 * a1 + ps[0][2] + ps[0][3] + ps[1][2] + ps[1][3];
#pragma unroll
    for (int i2 = 0; i2 < D / 8; ++i2) {
      o[i2][0] *= a0;
      o[i2][1] *= a0;
      o[i2][2] *= a1;
      o[i2][3] *= a1;
    }
    // P (bf16) as the A operand of O += P V: the C layout of S is the A layout
    uint32_t pa[4];
    pa[0] = pack_bf16x2(ps[0][0], ps[0][1]);
    pa[1] = pack_bf16x2(ps[0][2], ps[0][3]);
    pa[2] = pack_bf16x2(ps[1][0], ps[1][1]);
    pa[3] = pack_bf16x2(ps[1][2], ps[1][3]);
#pragma unroll
    for (int dn = 0; dn < D / 8; dn += 2) {
      const int r = (lane & 7) + ((lane >> 3) & 1) * 8;
      const int u = dn + (lane >> 4);
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(vb + swz<D>(r, u) * 16, b0, b1, b2, b3);
      mma_bf16(o[dn], pa, b0, b1);
      mma_bf16(o[dn + 1], pa, b2, b3);
    }
    __syncwarp();
  }
  cp_async_wait<0>();
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  __syncthreads();  // every warp is done with its stages: reuse them as merge scratch

  // ---- merge the 4 warp states: scratch[w] = { m[16], l[16], O[16][D] } ----
  float* scratch = reinterpret_cast<float*>(smem);
  constexpr int kWs = 32 + 16 * D;
  {
    float* ws = scratch + warp * kWs;
    const int g = lane >> 2, t2 = (lane & 3) * 2;
    if ((lane & 3) == 0) {
      ws[g] = m0;
      ws[g + 8] = m1;
      ws[16 + g] = l0;
      ws[16 + g + 8] = l1;
    }
#pragma unroll
    for (int dn = 0; dn < D / 8; ++dn) {
      ws[32 + g * D + dn * 8 + t2] = o[dn][0];
      ws[32 + g * D + dn * 8 + t2 + 1] = o[dn][1];
      ws[32 + (g + 8) * D + dn * 8 + t2] = o[dn][2];
      ws[32 + (g + 8) * D + dn * 8 + t2 + 1] = o[dn][3];
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < rows_valid * D; idx += kWarps * 32) {
    const int r = idx / D, c = idx % D;
    float mstar = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) mstar = fmaxf(mstar, scratch[w * kWs + r]);
    float acc = 0.f, lsum = 0.f;
    if (mstar != -CUDART_INF_F) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float f = ex2(scratch[w * kWs + r] - mstar);
        acc += f * scratch[w * kWs + 32 + r * D + c];
        lsum += f * scratch[w * kWs + 16 + r];
      }
    }
    const size_t prow = prow0 + (size_t)r * p.num_splits;
    p.o_part[prow * D + c] = lsum > 0.f ? acc / lsum : 0.f;
    if (c == 0) p.lse_part[prow] = lsum > 0.f ? (mstar + log2f(lsum)) * kLn2 : -CUDART_INF_F;
  }
}

// Output rows of one (sequence, KV-head group) from its nvalid non-empty
// split partials: lse = ln sum_s e^{lse_s}, O = sum_s e^{lse_s - lse} O_s.
template <int D>
__device__ __forceinline__ void merge_group(const DecodeParams& p, int b, int h0, int rows_valid, int nvalid) {
  constexpr int C4 = D / 4;
  for (int idx = threadIdx.x; idx < rows_valid * C4; idx += kWarps * 32) {
    const int r = idx / C4, c = (idx - r * C4) * 4;
    const size_t prow = ((size_t)b * p.Hq + h0 + r) * p.num_splits;
    float m = -CUDART_INF_F;
    for (int sp = 0; sp < nvalid; ++sp) m = fmaxf(m, __ldcg(p.lse_part + prow + sp));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
    if (m != -CUDART_INF_F) {
#pragma unroll 4
      for (int sp = 0; sp < nvalid; ++sp) {
        const float ls = __ldcg(p.lse_part + prow + sp);
        const float w = ls == -CUDART_INF_F ? 0.f : ex2((ls - m) * kLog2e);
        const float4 v = __ldcg(reinterpret_cast<const float4*>(p.o_part + (prow + sp) * D + c));
        acc.x += w * v.x;
        acc.y += w * v.y;
        acc.z += w * v.z;
        acc.w += w * v.w;
        wsum += w;
      }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    uint2 pk;
    pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
    pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.o) + ((size_t)b * p.Hq + h0 + r) * D + c) = pk;
    if (p.lse && c == 0) p.lse[(size_t)b * p.Hq + h0 + r] = wsum > 0.f ? m + logf(wsum) : -CUDART_INF_F;
  }
}

template <int D, bool kPage16>
__global__ void __launch_bounds__(kWarps * 32) decode_kernel(const DecodeParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_item, s_last;
  const int G = p.Hq / p.Hkv;
  const int nsub = (G + 15) >> 4;
  const int groups_per_seq = p.Hkv * nsub;
  const int groups = p.B * groups_per_seq;
  const int total = p.num_splits * groups;
  const int cap = p.max_pages_per_seq * p.page_size;
  const int chunk_pages = (p.max_pages_per_seq + p.num_splits - 1) / p.num_splits;
  const long long span = (long long)chunk_pages * p.page_size;
  for (;;) {
    if (threadIdx.x == 0) s_item = atomicAdd(p.counters, 1);
    __syncthreads();
    const int item = s_item;
    __syncthreads();
    if (item < 0 || item >= total) break;  // (a negative index cannot come from a zeroed counter)
    // highest split first: the long sequences' far chunks start early, empty items go fast
    const int split = p.num_splits - 1 - item / groups;
    const int g = item - (item / groups) * groups;
    const int b = g / groups_per_seq;
    const int hg = g - b * groups_per_seq;
    const int hkv = hg / nsub, sub = hg - hkv * nsub;
    const int rows_valid = min(16, G - sub * 16);
    const int h0 = hkv * G + sub * 16;
    int L = __ldg(p.seqlens + b);
    if (L < 0 || L > cap) {
      if (threadIdx.x == 0 && split == 0) record_status(p.status, kStatusDeviceCheck);
      L = L < 0 ? 0 : cap;
    }
    const int nvalid = (int)((L + span - 1) / span);   // non-empty splits of this sequence
    const long long t0 = (long long)split * span;
    if (t0 >= L) {  // empty split: mark it, and a sequence with no key at all gets O = 0, lse = -inf
      if (threadIdx.x < rows_valid)
        p.lse_part[((size_t)b * p.Hq + h0 + threadIdx.x) * p.num_splits + split] = -CUDART_INF_F;
      if (split == 0) merge_group<D>(p, b, h0, rows_valid, 0);
      continue;
    }
    decode_split<D, kPage16>(p, smem, split, b, hkv, h0, rows_valid, (int)t0, (int)min((long long)L, t0 + span));
    // publish the partial, count it, and let the last split of the group merge
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(p.counters + 1 + g, 1) == nvalid - 1;
    __syncthreads();
    if (s_last) {
      __threadfence();
      merge_group<D>(p, b, h0, rows_valid, nvalid);
    }
  }
}

// One CTA per (sequence, head) row: the splits are shared among groups of
// threads, each thread owning 4 consecutive output elements.
__global__ void __launch_bounds__(128) merge_kernel(const MergeParams p) {
  __shared__ float red[128 * 4 + 128 + 32];
  const int row = blockIdx.x;
  const int S = p.S, d = p.d;
  const float* lp = p.lse_part + (size_t)row * S;
  // max over splits
  float m = -CUDART_INF_F;
  for (int s = threadIdx.x; s < S; s += 128) m = fmaxf(m, lp[s]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  if ((threadIdx.x & 31) == 0) red[128 * 4 + 128 + (threadIdx.x >> 5)] = m;
  __syncthreads();
  m = fmaxf(fmaxf(red[128 * 4 + 128 + 0], red[128 * 4 + 128 + 1]),
            fmaxf(red[128 * 4 + 128 + 2], red[128 * 4 + 128 + 3]));

  const int nthr_d = d / 4;
  const int ngroups = 128 / nthr_d;
  const int grp = threadIdx.x / nthr_d;
  const int c = (threadIdx.x % nthr_d) * 4;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  if (grp < ngroups && m != -CUDART_INF_F) {
    const float* op = p.o_part + (size_t)row * S * d + c;
    for (int s = grp; s < S; s += ngroups) {
      const float ls = lp[s];
      if (ls == -CUDART_INF_F) continue;  // empty split: no weight, row never read
      const float w = ex2((ls - m) * kLog2e);
      const float4 v = *reinterpret_cast<const float4*>(op + (size_t)s * d);
      acc.x += w * v.x;
      acc.y += w * v.y;
      acc.z += w * v.z;
      acc.w += w * v.w;
      wsum += w;
    }
  }
  if (grp < ngroups) {
    red[threadIdx.x * 4 + 0] = acc.x;
    red[threadIdx.x * 4 + 1] = acc.y;
    red[threadIdx.x * 4 + 2] = acc.z;
    red[threadIdx.x * 4 + 3] = acc.w;
    red[128 * 4 + threadIdx.x] = wsum;
  }
  __syncthreads();
  if (grp == 0) {
    float4 tot = make_float4(0.f, 0.f, 0.f, 0.f);
    float wt = 0.f;
    for (int g2 = 0; g2 < ngroups; ++g2) {
      const int t = g2 * nthr_d + threadIdx.x;
      tot.x += red[t * 4 + 0];
      tot.y += red[t * 4 + 1];
      tot.z += red[t * 4 + 2];
      tot.w += red[t * 4 + 3];
      wt += red[128 * 4 + t];
    }
    const float inv = wt > 0.f ? 1.f / wt : 0.f;
    tot.x *= inv;
    tot.y *= inv;
    tot.z *= inv;
    tot.w *= inv;
    if (p.out_bf16) {
      __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(p.o) + (size_t)row * d + c;
      uint2 pk;
      pk.x = pack_bf16x2(tot.x, tot.y);
      pk.y = pack_bf16x2(tot.z, tot.w);
      *reinterpret_cast<uint2*>(ob) = pk;
    } else {
      *reinterpret_cast<float4*>(static_cast<float*>(p.o) + (size_t)row * d + c) = tot;
    }
    if (p.lse && threadIdx.x == 0) p.lse[row] = wt > 0.f ? m + logf(wt) : -CUDART_INF_F;
  }
}

template <int D, bool kPage16>
cudaError_t launch_decode_t(const DecodeParams& p, cudaStream_t stream) {
  using Lay = DecodeLayout<D>;
  auto kern = decode_kernel<D, kPage16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Lay::kBytes);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kWarps * 32, Lay::kBytes);
  if (e != cudaSuccess) return e;
  const int sms = num_sms_current();
  if (sms <= 0 || per_sm <= 0) return cudaErrorInvalidValue;
  // work counter + one arrival counter per (sequence, KV-head group) start at zero
  e = cudaMemsetAsync(p.counters, 0, (size_t)(1 + p.B * p.Hq) * sizeof(int), stream);
  if (e != cudaSuccess) return e;
  const int G = p.Hq / p.Hkv;
  const long long items = (long long)p.num_splits * p.B * p.Hkv * ((G + 15) / 16);
  const long long slots = (long long)sms * per_sm;
  const int grid = (int)(items < slots ? items : slots);
  kern<<<grid, kWarps * 32, Lay::kBytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream) {
  const bool p16 = p.page_size == 16;
  if (p.d == 128) return p16 ? launch_decode_t<128, true>(p, stream) : launch_decode_t<128, false>(p, stream);
  return p16 ? launch_decode_t<64, true>(p, stream) : launch_decode_t<64, false>(p, stream);
}

cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream) {
  merge_kernel<<<p.B * p.Hq, 128, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace fattn
