// libfattn C ABI: argument validation, the device status word, TMA
// descriptor encoding and kernel dispatch. See include/fattn.h for the
// contract of every entry point.
#include "fattn.h"
#include "fattn_internal.h"

#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <mutex>

namespace fattn {

// First device-side problem since the last fattn_debug_read_status().
__device__ int g_status_word = 0;

static std::atomic<int*> g_status_ptr[128];

// Test hook of the bounded pipeline waits (fattn_debug_set_wait_limit): the limit of
// every wait of later tensor-core launches (0 = kDefaultWaitNs) and the stall flag.
static std::atomic<unsigned long long> g_wait_limit_ns{0};
static std::atomic<int> g_debug_stall{0};

template <typename Params>
void set_waits(Params& p) {
  const unsigned long long w = g_wait_limit_ns.load(std::memory_order_relaxed);
  p.wait_ns = w ? w : kDefaultWaitNs;
  p.debug_stall = g_debug_stall.load(std::memory_order_relaxed);
}

int* status_ptr(int* err) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) {
    *err = 1;
    return nullptr;
  }
  int* p = g_status_ptr[dev].load(std::memory_order_acquire);
  if (p) return p;
  void* addr = nullptr;
  if (cudaGetSymbolAddress(&addr, g_status_word) != cudaSuccess || addr == nullptr) {
    *err = 1;
    return nullptr;
  }
  g_status_ptr[dev].store(static_cast<int*>(addr), std::memory_order_release);
  return static_cast<int*>(addr);
}

static PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 3-D bf16 view [rows, H, d] (d innermost) with a box of box_rows x 1 head x
// 64 elements (128 bytes, the 128-byte swizzle span). Rows past `rows` read as
// zero.
bool encode_rows_map(CUtensorMap* map, const void* base, int rows, int H, int d, int box_rows) {
  auto fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D view of one-byte elements (E4M3) [d2][d1][d0] with row strides s1, s2
// (bytes), box b0 x b1 x b2, 128-byte swizzle. Elements past the view read as zero.
bool encode_u8_map(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1,
                   uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2) {
  auto fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {s1, s2};
  cuuint32_t box[3] = {b0, b1, b2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int num_sms_current() {  // declared in fattn_internal.h
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

}  // namespace fattn

using namespace fattn;

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

extern "C" const char* fattn_status_string(fattn_status s) {
  switch (s) {
    case FATTN_OK: return "ok";
    case FATTN_ERR_INVALID_ARG: return "invalid argument";
    case FATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case FATTN_ERR_WORKSPACE: return "workspace missing or too small";
    case FATTN_ERR_CUDA: return "CUDA error";
    case FATTN_ERR_TIMEOUT: return "device pipeline wait timed out";
    case FATTN_ERR_DEVICE_CHECK: return "device-side index check failed";
  }
  return "unknown status";
}

extern "C" fattn_status fattn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                                  int Hkv, int N, int d, int causal, float scale, const int32_t* cu_seqlens,
                                  int total_tokens, fattn_dtype dtype, cudaStream_t stream) {
  if (B < 0 || N < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || total_tokens < 0) return FATTN_ERR_INVALID_ARG;
  // An empty problem is valid whatever the pointers (an empty tensor may have none).
  if (B == 0 || N == 0 || (cu_seqlens && total_tokens == 0)) return FATTN_OK;
  if (!q || !k || !v || !o) return FATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return FATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return FATTN_ERR_INVALID_ARG;
  if (dtype != FATTN_BF16 && dtype != FATTN_FP32) return FATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return FATTN_ERR_INVALID_ARG;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return FATTN_ERR_INVALID_ARG;
  if (cu_seqlens && (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u)) return FATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FATTN_ERR_UNSUPPORTED;
  const long long rows = cu_seqlens ? (long long)total_tokens : (long long)B * N;
  if (rows > 0x7fffffffLL || (long long)B * Hq * N > 0x7fffffffLL * 4LL) return FATTN_ERR_UNSUPPORTED;

  int err = 0;
  PrefillParams p{};  // no block mask, no block table
  p.mask_heads = 1;
  p.q = q; p.k = k; p.v = v; p.o = o; p.lse = lse; p.cu_seqlens = cu_seqlens;
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.N = N; p.d = d; p.total_rows = (int)rows;
  p.causal = causal ? 1 : 0; p.scale = scale;
  p.status = status_ptr(&err);
  if (err) return FATTN_ERR_CUDA;
  set_waits(p);

  cudaError_t e;
  if (dtype == FATTN_FP32) {
    e = launch_prefill_f32(p, stream);
  } else {
    CUtensorMap tq, tk, tv, to;
    if (!encode_rows_map(&tq, q, p.total_rows, Hq, d, 128) || !encode_rows_map(&tk, k, p.total_rows, Hkv, d, 128) ||
        !encode_rows_map(&tv, v, p.total_rows, Hkv, d, 128) || !encode_rows_map(&to, o, p.total_rows, Hq, d, 32))
      return FATTN_ERR_CUDA;
    int sms = num_sms_current();
    if (sms <= 0) return FATTN_ERR_CUDA;
    e = launch_prefill_tc(p, tq, tk, tv, to, sms, stream);
  }
  return e == cudaSuccess ? FATTN_OK : FATTN_ERR_CUDA;
}

extern "C" fattn_status fattn_fwd_block_sparse(const void* q, const void* k, const void* v, void* o, float* lse,
                                               int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                                               const uint8_t* block_mask, int mask_heads, cudaStream_t stream) {
  if (B < 0 || N < 0 || Hq <= 0 || Hkv <= 0 || d <= 0) return FATTN_ERR_INVALID_ARG;
  if (B == 0 || N == 0) return FATTN_OK;
  if (!q || !k || !v || !o || !block_mask) return FATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0 || (mask_heads != 1 && mask_heads != Hq)) return FATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return FATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return FATTN_ERR_INVALID_ARG;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return FATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FATTN_ERR_UNSUPPORTED;
  static_assert(FATTN_SPARSE_MAX_BLOCKS == kSparseMaxBlocks, "mask row limit");
  if ((N + FATTN_SPARSE_BLOCK - 1) / FATTN_SPARSE_BLOCK > FATTN_SPARSE_MAX_BLOCKS) return FATTN_ERR_UNSUPPORTED;
  const long long rows = (long long)B * N;
  if (rows > 0x7fffffffLL) return FATTN_ERR_UNSUPPORTED;

  int err = 0;
  PrefillParams p{};
  p.q = q; p.k = k; p.v = v; p.o = o; p.lse = lse; p.cu_seqlens = nullptr;
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.N = N; p.d = d; p.total_rows = (int)rows;
  p.causal = causal ? 1 : 0; p.scale = scale;
  p.block_mask = block_mask;
  p.mask_heads = mask_heads;
  p.status = status_ptr(&err);
  if (err) return FATTN_ERR_CUDA;
  set_waits(p);
  CUtensorMap tq, tk, tv, to;
  if (!encode_rows_map(&tq, q, p.total_rows, Hq, d, 128) || !encode_rows_map(&tk, k, p.total_rows, Hkv, d, 128) ||
      !encode_rows_map(&tv, v, p.total_rows, Hkv, d, 128) || !encode_rows_map(&to, o, p.total_rows, Hq, d, 32))
    return FATTN_ERR_CUDA;
  const int sms = num_sms_current();
  if (sms <= 0) return FATTN_ERR_CUDA;
  return launch_prefill_tc(p, tq, tk, tv, to, sms, stream) == cudaSuccess ? FATTN_OK : FATTN_ERR_CUDA;
}

extern "C" fattn_status fattn_fwd_masked(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                                         int Hq, int Hkv, int N, int d, int causal, float scale, const void* mask,
                                         long long mask_batch_stride, long long mask_head_stride,
                                         int mask_row_stride, cudaStream_t stream) {
  if (B < 0 || N < 0 || Hq <= 0 || Hkv <= 0 || d <= 0) return FATTN_ERR_INVALID_ARG;
  if (B == 0 || N == 0) return FATTN_OK;
  if (!q || !k || !v || !o || !mask) return FATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0 || !std::isfinite(scale)) return FATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(mask)) return FATTN_ERR_INVALID_ARG;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return FATTN_ERR_INVALID_ARG;
  // whole 16-byte groups of 8 entries: every stride a multiple of 8, rows at least N long
  if (mask_row_stride < N || mask_row_stride % 8 || mask_batch_stride < 0 || mask_batch_stride % 8 ||
      mask_head_stride < 0 || mask_head_stride % 8)
    return FATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FATTN_ERR_UNSUPPORTED;
  const long long rows = (long long)B * N;
  if (rows > 0x7fffffffLL) return FATTN_ERR_UNSUPPORTED;

  int err = 0;
  PrefillParams p{};
  p.q = q; p.k = k; p.v = v; p.o = o; p.lse = lse; p.cu_seqlens = nullptr;
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.N = N; p.d = d; p.total_rows = (int)rows;
  p.causal = causal ? 1 : 0; p.scale = scale;
  p.mask_heads = 1;
  p.mask = mask; p.mask_sb = mask_batch_stride; p.mask_sh = mask_head_stride; p.mask_ld = mask_row_stride;
  p.mask_v8 = (reinterpret_cast<uintptr_t>(mask) & 31u) == 0 && mask_row_stride % 16 == 0 &&
              mask_batch_stride % 16 == 0 && mask_head_stride % 16 == 0;
  p.status = status_ptr(&err);
  if (err) return FATTN_ERR_CUDA;
  set_waits(p);
  CUtensorMap tq, tk, tv, to;
  if (!encode_rows_map(&tq, q, p.total_rows, Hq, d, 128) || !encode_rows_map(&tk, k, p.total_rows, Hkv, d, 128) ||
      !encode_rows_map(&tv, v, p.total_rows, Hkv, d, 128) || !encode_rows_map(&to, o, p.total_rows, Hq, d, 32))
    return FATTN_ERR_CUDA;
  const int sms = num_sms_current();
  if (sms <= 0) return FATTN_ERR_CUDA;
  return launch_prefill_tc(p, tq, tk, tv, to, sms, stream) == cudaSuccess ? FATTN_OK : FATTN_ERR_CUDA;
}

extern "C" fattn_status fattn_fwd_paged(const void* q, const void* kcache, const void* vcache,
                                        const int32_t* block_table, const int32_t* seqlens_k,
                                        const int32_t* cu_seqlens_q, void* o, float* lse, int B, int Hq, int Hkv,
                                        int d, int page_size, int max_pages_per_seq, int num_pages, int total_q,
                                        int max_seqlen_q, int causal, float scale, cudaStream_t stream) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || total_q < 0 || max_seqlen_q < 0 || page_size <= 0 ||
      max_pages_per_seq <= 0 || num_pages <= 0)
    return FATTN_ERR_INVALID_ARG;
  if (B == 0 || total_q == 0 || max_seqlen_q == 0) return FATTN_OK;
  if (!q || !kcache || !vcache || !block_table || !seqlens_k || !cu_seqlens_q || !o) return FATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0 || !std::isfinite(scale)) return FATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(o)) return FATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(seqlens_k) & 3u) ||
      (reinterpret_cast<uintptr_t>(cu_seqlens_q) & 3u) || (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return FATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FATTN_ERR_UNSUPPORTED;
  if (page_size != 16 && page_size != 32 && page_size != 64 && page_size != 128) return FATTN_ERR_UNSUPPORTED;
  // pool rows, plus one box past the end for slots beyond a sequence's pages
  if ((long long)(num_pages + 1) * page_size > 0x7fffffffLL) return FATTN_ERR_UNSUPPORTED;
  if ((long long)max_pages_per_seq * page_size > 0x7fffffffLL || (long long)B * max_pages_per_seq > 0x7fffffffLL)
    return FATTN_ERR_UNSUPPORTED;

  int err = 0;
  PrefillParams p{};
  p.q = q; p.k = kcache; p.v = vcache; p.o = o; p.lse = lse; p.cu_seqlens = cu_seqlens_q;
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.N = max_seqlen_q; p.d = d; p.total_rows = total_q;
  p.causal = causal ? 1 : 0; p.scale = scale;
  p.mask_heads = 1;
  p.block_table = block_table; p.seqlens_k = seqlens_k;
  p.page_size = page_size; p.max_pages = max_pages_per_seq; p.num_pages = num_pages;
  p.status = status_ptr(&err);
  if (err) return FATTN_ERR_CUDA;
  set_waits(p);
  CUtensorMap tq, tk, tv, to;
  const int pool_rows = num_pages * page_size;
  if (!encode_rows_map(&tq, q, total_q, Hq, d, 128) || !encode_rows_map(&tk, kcache, pool_rows, Hkv, d, page_size) ||
      !encode_rows_map(&tv, vcache, pool_rows, Hkv, d, page_size) || !encode_rows_map(&to, o, total_q, Hq, d, 32))
    return FATTN_ERR_CUDA;
  const int sms = num_sms_current();
  if (sms <= 0) return FATTN_ERR_CUDA;
  return launch_prefill_tc(p, tq, tk, tv, to, sms, stream) == cudaSuccess ? FATTN_OK : FATTN_ERR_CUDA;
}

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

extern "C" fattn_status fattn_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                                      int Hkv, int N, int d, int causal, float scale, float q_descale,
                                      float k_descale, float v_descale, cudaStream_t stream) {
  if (B < 0 || N < 0 || Hq <= 0 || Hkv <= 0 || d <= 0) return FATTN_ERR_INVALID_ARG;
  if (B == 0 || N == 0) return FATTN_OK;
  if (!q || !k || !v || !o) return FATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0 || !std::isfinite(scale)) return FATTN_ERR_INVALID_ARG;
  if (!(q_descale > 0.f) || !(k_descale > 0.f) || !(v_descale > 0.f) || !std::isfinite(q_descale) ||
      !std::isfinite(k_descale) || !std::isfinite(v_descale))
    return FATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return FATTN_ERR_INVALID_ARG;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return FATTN_ERR_INVALID_ARG;
  if (d != 128) return FATTN_ERR_UNSUPPORTED;
  const long long rows = (long long)B * N;
  if (rows > 0x7fffffffLL) return FATTN_ERR_UNSUPPORTED;

  int err = 0;
  PrefillParams p{};
  p.q = q; p.k = k; p.v = v; p.o = o; p.lse = lse; p.cu_seqlens = nullptr;
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.N = N; p.d = d; p.total_rows = (int)rows;
  p.causal = causal ? 1 : 0;
  p.scale = scale * q_descale * k_descale;  // S = scale (q_descale Q8)(k_descale K8)^T
  p.mask_heads = 1;
  p.fp8 = 1;
  p.v_descale = v_descale;
  p.status = status_ptr(&err);
  if (err) return FATTN_ERR_CUDA;
  set_waits(p);
  CUtensorMap tq, tk, tv, to;
  if (!encode_u8_map(&tq, q, d, Hq, rows, (uint64_t)d, (uint64_t)Hq * d, 128, 1, 128) ||
      !encode_u8_map(&tk, k, d, Hkv, rows, (uint64_t)d, (uint64_t)Hkv * d, 128, 1, 128) ||
      !encode_u8_map(&tv, v, d, Hkv, rows, (uint64_t)d, (uint64_t)Hkv * d, 128, 1, 128) ||
      !encode_rows_map(&to, o, (int)rows, Hq, d, 32))
    return FATTN_ERR_CUDA;
  const int sms = num_sms_current();
  if (sms <= 0) return FATTN_ERR_CUDA;
  return launch_prefill_tc(p, tq, tk, tv, to, sms, stream) == cudaSuccess ? FATTN_OK : FATTN_ERR_CUDA;
}

extern "C" size_t fattn_bwd_workspace_size(int B, int Hq, int N) {
  if (B <= 0 || Hq <= 0 || N <= 0) return 0;
  const size_t npad = ((size_t)N + 127) / 128 * 128;
  return 2 * align256((size_t)B * Hq * npad * sizeof(float));
}

extern "C" fattn_status fattn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                                  const void* dout, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N,
                                  int d, int causal, float scale, void* workspace, size_t workspace_bytes,
                                  cudaStream_t stream) {
  if (B < 0 || N < 0 || Hq <= 0 || Hkv <= 0 || d <= 0) return FATTN_ERR_INVALID_ARG;
  if (B == 0 || N == 0) return FATTN_OK;
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv) return FATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0 || !std::isfinite(scale)) return FATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) || !aligned16(dq) ||
      !aligned16(dk) || !aligned16(dv) || (reinterpret_cast<uintptr_t>(lse) & 3u))
    return FATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FATTN_ERR_UNSUPPORTED;
  const long long rows = (long long)B * N;
  const long long npad = ((long long)N + 127) / 128 * 128;
  if (rows > 0x7fffffffLL || (long long)B * Hq * npad > 0x7fffffffLL) return FATTN_ERR_UNSUPPORTED;
  const size_t need = fattn_bwd_workspace_size(B, Hq, N);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return FATTN_ERR_WORKSPACE;

  int err = 0;
  BwdParams p{};
  p.q = q; p.k = k; p.v = v; p.o = o; p.dout = dout; p.lse = lse;
  p.dq = dq; p.dk = dk; p.dv = dv;
  p.ws_nl2 = static_cast<float*>(workspace);
  p.ws_d = reinterpret_cast<float*>(static_cast<char*>(workspace) + need / 2);
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.N = N; p.d = d; p.Npad = (int)npad;
  p.causal = causal ? 1 : 0; p.scale = scale;
  p.status = status_ptr(&err);
  if (err) return FATTN_ERR_CUDA;
  set_waits(p);
  CUtensorMap tq, tk, tv, tdo, tdk, tdv;
  if (!encode_rows_map(&tq, q, (int)rows, Hq, d, 128) || !encode_rows_map(&tk, k, (int)rows, Hkv, d, 128) ||
      !encode_rows_map(&tv, v, (int)rows, Hkv, d, 128) || !encode_rows_map(&tdo, dout, (int)rows, Hq, d, 128) ||
      !encode_rows_map(&tdk, dk, (int)rows, Hkv, d, 32) || !encode_rows_map(&tdv, dv, (int)rows, Hkv, d, 32))
    return FATTN_ERR_CUDA;
  const int sms = num_sms_current();
  if (sms <= 0) return FATTN_ERR_CUDA;
  return launch_backward(p, tq, tk, tv, tdo, tdk, tdv, sms, stream) == cudaSuccess ? FATTN_OK : FATTN_ERR_CUDA;
}

extern "C" size_t fattn_decode_workspace_size(int B, int Hq, int d, int num_splits) {
  if (B <= 0 || Hq <= 0 || d <= 0 || num_splits <= 0) return 0;
  size_t rows = (size_t)B * Hq * num_splits;
  return align256(rows * sizeof(float)) + align256(rows * d * sizeof(float)) +
         align256((size_t)(1 + B * Hq) * sizeof(int));
}

extern "C" fattn_status fattn_decode_paged(const void* q, const void* kcache, const void* vcache,
                                           const int32_t* block_table, const int32_t* seqlens, int num_splits,
                                           void* o, float* lse, int B, int Hq, int Hkv, int d, int page_size,
                                           int max_pages_per_seq, int num_pages, float scale, void* workspace,
                                           size_t workspace_bytes, cudaStream_t stream) {
  if (!q || !kcache || !vcache || !block_table || !seqlens || !o) return FATTN_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || page_size <= 0 || max_pages_per_seq <= 0 || num_pages <= 0 ||
      num_splits <= 0)
    return FATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return FATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return FATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(o)) return FATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(seqlens) & 3u))
    return FATTN_ERR_INVALID_ARG;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return FATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FATTN_ERR_UNSUPPORTED;
  if ((long long)max_pages_per_seq * page_size > 0x7fffffffLL) return FATTN_ERR_UNSUPPORTED;
  if ((long long)num_pages * page_size * Hkv * d > (1LL << 40)) return FATTN_ERR_UNSUPPORTED;
  if ((long long)B * Hq * num_splits > 0x7fffffffLL / 512) return FATTN_ERR_UNSUPPORTED;
  const size_t need = fattn_decode_workspace_size(B, Hq, d, num_splits);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return FATTN_ERR_WORKSPACE;

  int err = 0;
  DecodeParams p;
  p.q = q; p.kcache = kcache; p.vcache = vcache; p.block_table = block_table; p.seqlens = seqlens;
  const size_t rows = (size_t)B * Hq * num_splits;
  p.lse_part = static_cast<float*>(workspace);
  p.o_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + align256(rows * sizeof(float)));
  p.counters = reinterpret_cast<int*>(static_cast<char*>(workspace) + align256(rows * sizeof(float)) +
                                      align256(rows * d * sizeof(float)));
  p.o = o;
  p.lse = lse;
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.d = d; p.page_size = page_size; p.max_pages_per_seq = max_pages_per_seq;
  p.num_pages = num_pages; p.num_splits = num_splits; p.scale = scale;
  p.status = status_ptr(&err);
  if (err) return FATTN_ERR_CUDA;
  return launch_decode(p, stream) == cudaSuccess ? FATTN_OK : FATTN_ERR_CUDA;
}

extern "C" fattn_status fattn_merge_partials(const float* o_part, const float* lse_part, void* o, float* lse, int B,
                                             int Hq, int num_splits, int d, fattn_dtype out_dtype,
                                             cudaStream_t stream) {
  if (!o_part || !lse_part || !o) return FATTN_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || num_splits <= 0 || d <= 0) return FATTN_ERR_INVALID_ARG;
  if (out_dtype != FATTN_BF16 && out_dtype != FATTN_FP32) return FATTN_ERR_INVALID_ARG;
  if (!aligned16(o_part) || !aligned16(o) || (reinterpret_cast<uintptr_t>(lse_part) & 3u))
    return FATTN_ERR_INVALID_ARG;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return FATTN_ERR_INVALID_ARG;
  if (d % 4 != 0 || d > 512) return FATTN_ERR_UNSUPPORTED;
  if ((long long)B * Hq * num_splits * d > 0x7fffffffLL) return FATTN_ERR_UNSUPPORTED;
  MergeParams m;
  m.o_part = o_part; m.lse_part = lse_part; m.o = o; m.lse = lse;
  m.B = B; m.Hq = Hq; m.S = num_splits; m.d = d; m.out_bf16 = out_dtype == FATTN_BF16;
  return launch_merge(m, stream) == cudaSuccess ? FATTN_OK : FATTN_ERR_CUDA;
}

extern "C" fattn_status fattn_debug_read_status(cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return FATTN_ERR_CUDA;
  int err = 0;
  int* p = status_ptr(&err);
  if (err) return FATTN_ERR_CUDA;
  int h = 0, zero = 0;
  if (cudaMemcpy(&h, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return FATTN_ERR_CUDA;
  if (cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return FATTN_ERR_CUDA;
  return static_cast<fattn_status>(h);
}

extern "C" void fattn_debug_set_wait_limit(unsigned long long limit_ns, int stall) {
  g_wait_limit_ns.store(limit_ns, std::memory_order_relaxed);
  g_debug_stall.store(stall ? 1 : 0, std::memory_order_relaxed);
}
