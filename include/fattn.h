/*
 * fattn.h — C ABI of libfattn: exact tiled attention on GB300 (sm_103a).
 *
 * The library computes exact attention, O = softmax(Q K^T * scale + M) V, tile
 * by tile with the online-softmax (m, l, O) rescaling rule, so the N x N score
 * and probability matrices never reach device memory. Sources:
 *   [FA-LLM]   "FlashAttention" (LLM-inference guide, ch. 10): the formula;
 *              "The trick: tiles and an online softmax" (update rule);
 *              "Decode is a different problem" / "Flash-Decoding" (split-K
 *              partials merged with the same rule); family table rows
 *              "Flash-Decoding" and "Paged variants".
 *   [FA-PAPER] "FlashAttention, explained": "The forward pass" steps 1-5
 *              (inputs Q, K, V of N x d per head in device memory, scale and
 *              mask fused, output O plus the per-row statistics l and m).
 *   [CUDA-OPS] "Attention" CUDA operations guide: K/V heads shared by several
 *              Q heads; non-contiguous (paged) KV allocation.
 *
 * Conventions shared by every call:
 *   - All tensor pointers are DEVICE pointers, owned by the caller, row-major,
 *     densely packed in the layout stated per call, and 16-byte aligned. The
 *     library never allocates, frees or synchronises on these calls.
 *   - Every call validates its arguments on the host first. On failure it
 *     returns a status and launches nothing; no call aborts or throws.
 *   - Work is enqueued on `stream` (0 = legacy default stream). A launch
 *     failure returns FATTN_ERR_CUDA. Problems found on the device (a
 *     block-table entry outside the pool, a sequence longer than its table,
 *     inconsistent cu_seqlens, a pipeline wait that did not finish within its
 *     time limit) are recorded in a device status word and the offending work
 *     is skipped; fattn_debug_read_status() reads and clears that word.
 *   - Query head h reads KV head h / (Hq / Hkv) (GQA; MQA when Hkv = 1).
 *   - lse is the natural-log logsumexp of the scaled, masked scores of a row,
 *     lse = m + ln(l); a row with no visible key has O = 0, lse = -inf.
 *   - Supported head dimensions: d = 64 and d = 128.
 */
#ifndef FATTN_H
#define FATTN_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FATTN_OK = 0,
  FATTN_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size, Hq % Hkv != 0 */
  FATTN_ERR_UNSUPPORTED = 2,   /* valid request outside the supported set (e.g. d = 96) */
  FATTN_ERR_WORKSPACE = 3,     /* workspace missing or smaller than required */
  FATTN_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed */
  FATTN_ERR_TIMEOUT = 5,       /* device status: a bounded pipeline wait expired */
  FATTN_ERR_DEVICE_CHECK = 6   /* device status: an index check failed, work skipped */
} fattn_status;

typedef enum {
  FATTN_BF16 = 0,
  FATTN_FP32 = 1
} fattn_dtype;

/*
 * fattn_fwd — prefill: exact attention for all query rows of a batch.
 * [FA-PAPER] "The forward pass"; [FA-LLM] formula and "The trick".
 *
 * Dense (cu_seqlens == NULL): q [B, N, Hq, d], k and v [B, N, Hkv, d],
 *   o [B, N, Hq, d] (same dtype as q), lse [B, Hq, N] fp32.
 * Varlen (cu_seqlens != NULL): B sequences packed back to back;
 *   cu_seqlens is a DEVICE int32 array [B + 1] with cu_seqlens[0] = 0,
 *   non-decreasing, cu_seqlens[B] = total_tokens; q [T, Hq, d], k and v
 *   [T, Hkv, d], o [T, Hq, d], lse [Hq, T] with T = total_tokens; N must be
 *   >= every sequence length (it sizes the launch; the host never reads
 *   cu_seqlens). No attention crosses a sequence boundary.
 * causal != 0 applies M = -inf above the diagonal of each sequence
 *   (key j visible to query i iff j <= i).
 * scale multiplies Q K^T (1/sqrt(d) is the usual choice); must be finite.
 * dtype: FATTN_BF16 runs the tensor-core kernel (fp32 accumulation, P rounded
 *   to bf16 for the P V product, O rounded to nearest even); FATTN_FP32 runs
 *   the CUDA-core fp32 kernel (inputs and outputs fp32).
 * lse may be NULL (not written). B == 0, N == 0 or total_tokens == 0 is an
 * empty problem: FATTN_OK, nothing launched.
 * Errors: INVALID_ARG for null q/k/v/o, negative sizes, Hq % Hkv != 0,
 *   non-finite scale, misaligned pointers; UNSUPPORTED for d not in {64, 128}.
 */
fattn_status fattn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                       int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                       const int32_t* cu_seqlens, int total_tokens,
                       fattn_dtype dtype, cudaStream_t stream);

/*
 * fattn_fwd_block_sparse — prefill restricted by a fixed block mask.
 * [FA-PAPER] "Block-sparse FlashAttention": given a fixed mask over blocks,
 * every tile that is zero in the mask is skipped (its scores take no part in
 * the softmax); the causal skip of fattn_fwd is the special case.
 *
 * Dense layout and bf16 only: q [B, N, Hq, d], k and v [B, N, Hkv, d],
 * o [B, N, Hq, d], lse [B, Hq, N] (lse may be NULL).
 * block_mask: DEVICE uint8 [mask_heads, nb, nb] with nb = ceil(N /
 *   FATTN_SPARSE_BLOCK); entry (h, i, j) != 0 keeps keys [128 j, 128 j + 128)
 *   for queries [128 i, 128 i + 128) of query head h (mask_heads = 1: one mask
 *   for every head; mask_heads = Hq: one per query head). With causal != 0
 *   the causal rule applies on top. A row that keeps no key gets O = 0,
 *   lse = -inf. Blocks that are zero are never loaded or computed.
 * Errors: those of fattn_fwd, INVALID_ARG for a NULL block_mask or
 *   mask_heads not in {1, Hq}, UNSUPPORTED for nb > FATTN_SPARSE_MAX_BLOCKS
 *   (N > 262144).
 */
#define FATTN_SPARSE_BLOCK 128
#define FATTN_SPARSE_MAX_BLOCKS 2048
fattn_status fattn_fwd_block_sparse(const void* q, const void* k, const void* v, void* o, float* lse,
                                    int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                                    const uint8_t* block_mask, int mask_heads, cudaStream_t stream);

/*
 * fattn_fwd_masked — prefill with a general additive mask M.
 * [FA-LLM] the formula O = softmax(Q K^T / sqrt(d) + M) V ("The trick: tiles
 * and an online softmax": M is added to each score tile while it is on chip).
 *
 * Dense layout and bf16, as fattn_fwd: q, o [B, N, Hq, d]; k, v [B, N, Hkv, d];
 * lse [B, Hq, N] (may be NULL).
 * mask: DEVICE bf16; entry (b, h, i, j) (query head h, query i, key j) is
 *   mask[b * mask_batch_stride + h * mask_head_stride + i * mask_row_stride + j]
 *   (strides in elements; 0 shares one mask over the batch or the heads). It is
 *   added to the scaled scores; -inf removes the key. With causal != 0 the
 *   causal rule applies on top. A row left with no key gets O = 0, lse = -inf.
 *   Entries at keys >= N are not read.
 * Errors: those of fattn_fwd (bf16, d in {64, 128}); INVALID_ARG for a NULL or
 *   misaligned (16 bytes) mask, mask_row_stride < N, or a stride that is negative
 *   or not a multiple of 8.
 */
fattn_status fattn_fwd_masked(const void* q, const void* k, const void* v, void* o, float* lse,
                              int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                              const void* mask, long long mask_batch_stride, long long mask_head_stride,
                              int mask_row_stride, cudaStream_t stream);

/*
 * fattn_fwd_fp8 — prefill on FP8 (E4M3) q, k, v with per-tensor descales.
 * [FA-LLM] "The FlashAttention family" (FlashAttention-3: FP8 on the tensor
 * cores); the computation is fattn_fwd's on the dequantized inputs
 * Q = q_descale * q, K = k_descale * k, V = v_descale * v.
 *
 * Dense layout: q [B, N, Hq, d], k, v [B, N, Hkv, d] as E4M3 bytes ('fn'
 * variant: no infinities); o [B, N, Hq, d] bf16; lse [B, Hq, N] fp32 (may be
 * NULL). Both products run on E4M3 operands with fp32 accumulation; P is
 * rounded to E4M3 for P V (the row sums use the unrounded P). V is read in
 * place (no copy, no workspace).
 * Errors: INVALID_ARG (NULL or misaligned pointers, negative sizes,
 *   Hq % Hkv != 0, a descale that is not finite and positive), UNSUPPORTED
 *   (d != 128, B * N >= 2^31).
 */
fattn_status fattn_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse,
                           int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                           float q_descale, float k_descale, float v_descale, cudaStream_t stream);

/*
 * fattn_fwd_paged — prefill of query chunks against a paged KV cache
 * (chunked prefill, or a whole prompt read back from the cache).
 * [FA-LLM] "Paged variants" (the tiled computation with K/V read through a
 * block table); [FA-PAPER] "The forward pass" (the computation itself).
 *
 * q [total_q, Hq, d] bf16: B chunks packed back to back; chunk b is rows
 *   [cu_seqlens_q[b], cu_seqlens_q[b+1]) (Lq_b rows) and holds the queries of
 *   the LAST Lq_b positions of sequence b's context.
 * kcache, vcache [num_pages, page_size, Hkv, d] bf16: token t of sequence b is
 *   slot t % page_size of page block_table[b * max_pages_per_seq + t / page_size].
 * seqlens_k [B] int32, cu_seqlens_q [B + 1] int32, block_table int32: DEVICE.
 *   seqlens_k[b] counts the context tokens including the chunk's own:
 *   Lq_b <= seqlens_k[b] <= max_pages_per_seq * page_size.
 * o [total_q, Hq, d] bf16; lse [Hq, total_q] fp32 (may be NULL).
 * causal != 0: query i of chunk b sees keys j <= i + seqlens_k[b] - Lq_b.
 * max_seqlen_q: host upper bound on every Lq_b (sizes the grid).
 * Supported: d in {64, 128}, page_size in {16, 32, 64, 128}.
 * Slots past seqlens_k[b] in a sequence's last page are read and get weight 0,
 *   so they must hold finite values; table entries past the last page are not read.
 * Errors: INVALID_ARG (NULL or misaligned pointers, negative sizes,
 *   Hq % Hkv != 0, non-finite scale); UNSUPPORTED (d, page_size,
 *   (num_pages + 1) * page_size >= 2^31). A table entry outside
 *   [0, num_pages) (read as zeros), a seqlens_k outside the range above or a
 *   bad cu_seqlens_q (chunk skipped) record FATTN_ERR_DEVICE_CHECK in the
 *   status word.
 */
fattn_status fattn_fwd_paged(const void* q, const void* kcache, const void* vcache,
                             const int32_t* block_table, const int32_t* seqlens_k,
                             const int32_t* cu_seqlens_q, void* o, float* lse,
                             int B, int Hq, int Hkv, int d, int page_size, int max_pages_per_seq,
                             int num_pages, int total_q, int max_seqlen_q, int causal, float scale,
                             cudaStream_t stream);

/*
 * fattn_bwd_workspace_size — bytes of scratch fattn_bwd needs: two fp32
 * arrays [B * Hq, Npad] (Npad = N rounded up to 128), each 256-byte aligned.
 * Returns 0 for non-positive arguments.
 */
size_t fattn_bwd_workspace_size(int B, int Hq, int N);

/*
 * fattn_bwd — gradients of attention with respect to q, k and v.
 * [FA-PAPER] "The backward pass recomputes instead of reading": P is rebuilt
 * tile by tile from the saved logsumexp; D = rowsum(dO o O), dV = P^T dO,
 * dP = dO V^T, dS = P o (dP - D), dQ = scale dS K, dK = scale dS^T Q.
 *
 * Dense layout, bf16: q, o, dout, dq [B, N, Hq, d]; k, v, dk, dv
 * [B, N, Hkv, d]; lse [B, Hq, N] fp32 as written by fattn_fwd for the same
 * q, k, v, causal and scale (o likewise). dk and dv sum over the Hq / Hkv
 * query heads that share a KV head. All buffers are DEVICE memory.
 * workspace: DEVICE, >= fattn_bwd_workspace_size(B, Hq, N) bytes, 256-byte
 *   aligned, contents ignored; owned by the caller.
 * Errors: INVALID_ARG (NULL or misaligned pointers, negative sizes,
 *   Hq % Hkv != 0, non-finite scale), UNSUPPORTED (d not in {64, 128},
 *   B * N or B * Hq * Npad >= 2^31), WORKSPACE (missing, small or misaligned).
 */
fattn_status fattn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                       const void* dout, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N, int d,
                       int causal, float scale, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * fattn_decode_workspace_size — bytes of scratch fattn_decode_paged needs:
 * the per-split partials lse_part [B, Hq, S] fp32 and o_part [B, Hq, S, d]
 * fp32 (S = num_splits), then 1 + B * Hq int32 work-scheduling counters, each
 * region 256-byte aligned. Returns 0 for non-positive arguments.
 */
size_t fattn_decode_workspace_size(int B, int Hq, int d, int num_splits);

/*
 * fattn_decode_paged — split-KV decode over a paged KV cache.
 * [FA-LLM] "Decode is a different problem", "Flash-Decoding" (split the KV
 * sequence across thread blocks, merge the partial (m, l, O) with the same
 * online-softmax rule) and "Paged variants" (read K/V through a block table).
 *
 * q [B, Hq, d] bf16: one query token per sequence, which sees all seqlens[b]
 *   keys of its sequence.
 * kcache, vcache [num_pages, page_size, Hkv, d] bf16: the shared page pool.
 * block_table DEVICE int32 [B, max_pages_per_seq]: logical page p of sequence
 *   b is pool page block_table[b * max_pages_per_seq + p]. Entries past a
 *   sequence's last page are never read.
 * seqlens DEVICE int32 [B]: context length of each sequence, 0 <= seqlens[b]
 *   <= max_pages_per_seq * page_size.
 * num_splits = S >= 1: every sequence's pages are cut into S chunks of
 *   C = ceil(max_pages_per_seq / S) whole pages; split s covers tokens
 *   [s*C*page_size, min(seqlens[b], (s+1)*C*page_size)) and is empty past
 *   the end of the sequence.
 * o [B, Hq, d] bf16, lse [B, Hq] fp32 (lse may be NULL).
 * workspace: device scratch of at least fattn_decode_workspace_size(B, Hq, d,
 *   S) bytes, 256-byte aligned; its contents on entry do not matter (the call
 *   zeroes its counters with cudaMemsetAsync on `stream`). After the call it
 *   holds the partials (lse_part first, then o_part; each o_part row divided
 *   by its own l, and lse_part = -inf for an empty split). The partials are
 *   merged into o and lse inside the same kernel launch.
 * Errors: INVALID_ARG (null/misaligned pointers, non-positive sizes,
 *   Hq % Hkv != 0, non-finite scale), UNSUPPORTED (d not in {64, 128}),
 *   WORKSPACE (workspace NULL or too small). A block-table entry outside
 *   [0, num_pages) or a seqlens entry above the table's capacity is caught on
 *   the device: the affected pages are skipped and FATTN_ERR_DEVICE_CHECK is
 *   recorded in the status word.
 */
fattn_status fattn_decode_paged(const void* q, const void* kcache, const void* vcache,
                                const int32_t* block_table, const int32_t* seqlens,
                                int num_splits, void* o, float* lse,
                                int B, int Hq, int Hkv, int d, int page_size,
                                int max_pages_per_seq, int num_pages, float scale,
                                void* workspace, size_t workspace_bytes,
                                cudaStream_t stream);

/*
 * fattn_merge_partials — merge split partials with the online-softmax rule.
 * [FA-LLM] "Flash-Decoding": each chunk's partial (m, l, O) is merged with
 * the same rescaling rule.
 *
 * o_part [B, Hq, S, d] fp32 holds each split's output already divided by its
 * own l; lse_part [B, Hq, S] fp32 its logsumexp (-inf = empty split, whose
 * o_part row is never read). Output: lse = ln(sum_s e^{lse_s}),
 * O = sum_s e^{lse_s - lse} O_s, written to o [B, Hq, d] in out_dtype and lse
 * [B, Hq] fp32 (lse may be NULL). All splits empty gives O = 0, lse = -inf.
 * Errors: INVALID_ARG (null/misaligned pointers, non-positive sizes),
 * UNSUPPORTED (d not a positive multiple of 4 up to 512).
 */
fattn_status fattn_merge_partials(const float* o_part, const float* lse_part, void* o, float* lse,
                                  int B, int Hq, int num_splits, int d, fattn_dtype out_dtype,
                                  cudaStream_t stream);

/*
 * fattn_decode_paged_static — fattn_decode_paged without a workspace, for
 * callers that cannot allocate device memory. The pages have no counterpart:
 * this is library plumbing. Some callers cannot call cudaMalloc: plugins whose
 * host (an inference server or another runtime) hands them only their input
 * and output buffers, and code that must stay inside a device-memory budget
 * owned by a pool it cannot draw from. This call runs the same kernels as
 * fattn_decode_paged, with the split partials kept in a fixed scratch array
 * of FATTN_DECODE_STATIC_SCRATCH_BYTES (32 MiB) that is part of the library's
 * device image: every GPU that loads the library holds it until the process
 * exits. The call allocates and frees nothing.
 *
 * Arguments, layouts and outputs are those of fattn_decode_paged minus the
 * workspace. The first call on a device (with that device current) looks up
 * the scratch's device address with cudaGetSymbolAddress and caches it; make
 * that first call before any stream capture on that device. All calls share
 * the one scratch array, which keeps the last call's contents; each call
 * zeroes the counters it uses (cudaMemsetAsync on `stream`) and reads back
 * only partials it wrote itself. Calls that overlap on the GPU — on different
 * streams, or from different host threads — race on the array and must be
 * serialised by the caller.
 * Errors: those of fattn_decode_paged; FATTN_ERR_WORKSPACE when the partials
 * (fattn_decode_workspace_size(B, Hq, d, num_splits) bytes) exceed the
 * scratch; FATTN_ERR_CUDA if the scratch address cannot be obtained.
 */
#define FATTN_DECODE_STATIC_SCRATCH_BYTES ((size_t)32 << 20)
fattn_status fattn_decode_paged_static(const void* q, const void* kcache, const void* vcache,
                                       const int32_t* block_table, const int32_t* seqlens,
                                       int num_splits, void* o, float* lse,
                                       int B, int Hq, int Hkv, int d, int page_size,
                                       int max_pages_per_seq, int num_pages, float scale,
                                       cudaStream_t stream);

/* Static English description of a status code (never NULL). */
const char* fattn_status_string(fattn_status status);

/*
 * fattn_debug_read_status — synchronise `stream`, then read and clear the
 * device status word of the current device. Returns FATTN_OK if no device-side
 * check failed since the last read, else the first recorded code
 * (FATTN_ERR_TIMEOUT or FATTN_ERR_DEVICE_CHECK), or FATTN_ERR_CUDA if the
 * synchronisation itself failed. Meant for tests and debugging: it blocks.
 */
fattn_status fattn_debug_read_status(cudaStream_t stream);

/*
 * fattn_debug_set_wait_limit — test hook for the bounded pipeline waits of the
 * tensor-core kernels (every prefill variant and the backward passes; decode and
 * the fp32 prefill have no such waits). The pages have no counterpart: this is
 * library plumbing for failure tests.
 *
 * Every mbarrier wait of those kernels gives up after a limit (default 2 s):
 * it records FATTN_ERR_TIMEOUT in the device status word, every role of the
 * kernel stops, copies and tensor-core products already issued are waited for,
 * TMEM is freed and the kernel returns, so the CUDA context stays usable.
 * limit_ns > 0 sets that limit for launches made after this call (0 restores the
 * default). stall != 0 makes the softmax / element-wise warps of those launches
 * first wait on a barrier that no role ever arrives on, so the wait runs out after
 * limit_ns: the launch then writes none of its outputs and the status word reads
 * FATTN_ERR_TIMEOUT. The setting is process-wide and not synchronised with
 * launches in flight on other host threads; reset it with (0, 0).
 */
void fattn_debug_set_wait_limit(unsigned long long limit_ns, int stall);

#ifdef __cplusplus
}
#endif

#endif /* FATTN_H */
