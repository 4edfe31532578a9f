// Internal launchers of libfattn (not part of the ABI). Each returns a
// cudaError_t from the launch; argument checks happen in api.cu before these
// are called.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fattn {

// Device status word codes (match fattn_status).
enum : int { kStatusOk = 0, kStatusTimeout = 5, kStatusDeviceCheck = 6 };

// Limit of one pipeline wait unless a test sets another (fattn_debug_set_wait_limit).
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;

// Problem description shared by both prefill kernels.
struct PrefillParams {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  const int32_t* cu_seqlens;  // device; nullptr = dense
  int B, Hq, Hkv, N, d;       // N = sequence length (dense) / max length (varlen)
  int total_rows;             // rows of the packed [rows, H, d] view (B*N or T)
  int causal;
  float scale;
  int* status;                // device status word
  // block-sparse variant only: uint8 [mask_heads][nb][nb], nb = ceil(N / 128);
  // block (qb, kb) = 0 hides keys [128 kb, 128 kb + 128) from queries [128 qb, 128 qb + 128)
  const uint8_t* block_mask;  // nullptr = dense
  int mask_heads;             // 1 (shared by all heads) or Hq
  // paged variant only (K/V read through a block table; q, o, lse packed as in
  // varlen with cu_seqlens = the chunks' query offsets):
  const int32_t* block_table; // device [B][max_pages]; nullptr = K/V in q's row space
  const int32_t* seqlens_k;   // device [B]: context tokens per sequence (>= its queries)
  int page_size, max_pages, num_pages;
  // masked variant only: additive bf16 mask, entry (b, h, i, j) at
  // mask[b * mask_sb + h * mask_sh + i * mask_ld + j] (strides in elements, multiples of 8)
  const void* mask;           // nullptr = none
  long long mask_sb, mask_sh;
  int mask_ld;
  int mask_v8;                // the mask is 32-byte aligned and its strides are multiples of 16
                              // elements: rows are read with 32-byte loads
  // FP8 variant only: E4M3 q, k and v ([rows, H, d]); scale already holds
  // scale * q_descale * k_descale
  int fp8;
  float v_descale;
  // bounded pipeline waits: each mbarrier wait gives up after wait_ns; debug_stall != 0
  // (test hook) makes the softmax / element-wise warps first wait on a barrier that no
  // role arrives on, so that the wait runs out and every role takes the abort exit
  unsigned long long wait_ns;
  int debug_stall;
};

// Longest mask row (blocks) the block-sparse kernel holds in shared memory.
constexpr int kSparseMaxBlocks = 2048;

// Tensor-core prefill (bf16 in, fp32 accumulate, bf16 out). Tensor maps are
// encoded by the caller over the packed [rows, H, d] views of q, k and v (128-row
// boxes) and of o (bf16, 32-row boxes: the epilogue's stores).
cudaError_t launch_prefill_tc(const PrefillParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                              const CUtensorMap& tv, const CUtensorMap& to, int num_sms, cudaStream_t stream);

// CUDA-core fp32 prefill.
cudaError_t launch_prefill_f32(const PrefillParams& p, cudaStream_t stream);

struct DecodeParams {
  const void* q;
  void* o;          // [B, Hq, d] bf16 output
  float* lse;       // [B, Hq] or nullptr
  int* counters;    // workspace: work counter, then one arrival counter per (sequence, KV-head group)
  const void* kcache;
  const void* vcache;
  const int32_t* block_table;
  const int32_t* seqlens;
  float* lse_part;  // [B, Hq, S]
  float* o_part;    // [B, Hq, S, d]
  int B, Hq, Hkv, d, page_size, max_pages_per_seq, num_pages, num_splits;
  float scale;
  int* status;
};

// Split-KV decode with the merge fused in (one launch, after a memset of the counters).
cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream);

int num_sms_current();

struct MergeParams {
  const float* o_part;
  const float* lse_part;
  void* o;
  float* lse;
  int B, Hq, S, d;
  int out_bf16;
};

cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream);

// Attention backward (dense [B, N, H, d] bf16, lse [B, Hq, N] fp32 from the forward).
struct BwdParams {
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const void* dout;
  const float* lse;
  void* dq;
  void* dk;
  void* dv;
  float* ws_nl2;              // [B * Hq, Npad]: -lse * log2(e), -inf past N
  float* ws_d;                // [B * Hq, Npad]: rowsum(dO o O), 0 past N
  int B, Hq, Hkv, N, d, Npad; // Npad = N rounded up to 128
  int causal;
  float scale;
  int* status;
  // bounded pipeline waits: each mbarrier wait gives up after wait_ns; debug_stall != 0
  // (test hook) makes the softmax / element-wise warps first wait on a barrier that no
  // role arrives on, so that the wait runs out and every role takes the abort exit
  unsigned long long wait_ns;
  int debug_stall;
};

// dQ pass (which also writes the workspace's two vectors) and dK/dV pass, in that
// order on `stream`. Tensor maps are over the packed [B * N, H, d] views of q, k, v
// and dout (128-row boxes) and of dk and dv (32-row boxes, for the stores).
cudaError_t launch_backward(const BwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const CUtensorMap& tdk, const CUtensorMap& tdv, int num_sms,
                            cudaStream_t stream);

}  // namespace fattn
