// Tensor-core prefill for sm_103a: exact attention tile by tile with the
// online-softmax rule ("The trick: tiles and an online softmax", FlashAttention
// LLM-inference page; "The forward pass", FlashAttention explained).
//
// One CTA per SM loops over work items (sequence, query head, 256 query rows =
// two 128-row Q tiles A and B that share every K/V tile). Roles:
//   warp 0      TMA producer: Q_A and Q_B once per item, then per step j the
//               tiles K_j and V_{j-1} into one slot of a ring (two slots; three
//               in the FP8 variant, whose tiles are half the size) under that
//               slot's full / empty barrier pair (128-byte swizzle, 64-column
//               boxes).
//   warp 1      MMA issuer (one thread). Per K/V tile j it issues
//               O_A += P_A(j-1) V_{j-1}, S_A = Q_A K_j^T, O_B += P_B(j-1) V_{j-1},
//               S_B = Q_B K_j^T, so that while one softmax warpgroup works on its
//               scores the tensor core runs the other tile's two products.
//   warps 2-3   complete the first warpgroup, which gives registers to the
//               softmax warpgroups with setmaxnreg; in the block-sparse variant
//               warp 2 reads the block mask ahead of the other roles.
//   warps 4-7   softmax of tile A, warps 8-11 softmax of tile B: each thread owns
//               one query row (TMEM lane); it loads its 128 scores, masks (causal
//               diagonal, sequence end), keeps the running max m and sum l in
//               registers, writes P (bf16) over the first 64 columns of its S
//               buffer, rescales O in TMEM when the max moved, and at the end
//               writes O / l (bf16) and lse = m + ln l. A warp whose 32 rows all
//               lie in the sequence stages them in shared memory and writes them
//               with TMA tensor stores (one 32-row box per 64 columns) instead of
//               one 256-byte row per thread, scattered over rows 8 KB apart.
// The running max is raised lazily: a row keeps its old m while no new score
// exceeds it by more than 2^8 (p <= 256 then, exact in the final O/l because O
// and l use the same m), which makes the O rescale rare.
// Causal tiles above the diagonal are never loaded or computed ("tiles above
// the diagonal are never touched"). S and P never leave the SM.
// Block-sparse variant ("Block-sparse FlashAttention": zero blocks of a fixed
// block mask are skipped): with 128 x 128 blocks, a tile visits only the K/V
// blocks its mask row keeps (highest first); warp 2 turns the item's two mask rows into bit
// words in a shared-memory ring, the producer and the MMA warp walk the union
// of the two tiles' kept blocks in the same interleaved order, each softmax
// warpgroup walks its own row, and a tile whose rows keep no block writes
// O = 0, lse = -inf.
// Paged variant ("Paged variants"): K/V tiles come page by page through the
// block table, eight producer lanes each issuing one page's box. Masked variant
// (the formula's additive M): each softmax thread adds its row's bf16 mask
// entries to the scaled scores, the first 64 keys of a tile by 32- or 16-byte
// loads into registers, the other 64 copied by the warp into its staging slot,
// both requested before the wait for the scores. FP8 variant (FlashAttention-3
// row of "The FlashAttention family"): E4M3 Q, K and V (kind::f8f6f4 products,
// V read in place as an MN-major operand), P rounded to E4M3 in shared memory.
//
// P_X aliases S_X: S_X(j) is issued right after O_X += P_X(j-1) V by the same
// thread, and tcgen05.mma operations issued by one thread execute in order, so
// the product has read P_X(j-1) before S_X(j) overwrites those columns. The
// softmax writes P_X(j) only after S_X(j) completed, whose commit covers every
// earlier MMA, O_X += P_X(j-1) V included.
// Where P_X has a buffer of its own (bf16 at d = 64: TMEM columns 384 and 448;
// the FP8 variant: shared memory), S_X(j) is issued as soon as the softmax has
// read S_X(j-1) into registers (barrier SFree), and the softmax waits for
// O_X += P_X(j-1) V to complete (barrier PvDone, one commit per product) before
// it rescales O_X or rewrites P_X; the epilogue waits for the last one.
//
// Every pipeline wait is bounded: a wait that exceeds its limit records
// FATTN_ERR_TIMEOUT in the device status word, every role stops, in-flight
// copies and MMAs are drained, TMEM is freed and the kernel returns.
#include "device_common.cuh"
#include "fattn_internal.h"
#include "sm100_primitives.cuh"

#include <cuda_fp8.h>
#include <math_constants.h>

namespace fattn {
namespace {

using namespace sm100;

constexpr int BM = 128;          // query rows per tile (M of one tcgen05.mma)
constexpr int BN = 128;          // keys per K/V tile
constexpr int kRowsPerItem = 2 * BM;
constexpr int kThreads = 384;    // 3 warpgroups
// Register split (setmaxnreg): launched at 168 per thread (65536 / 384, rounded
// down to the allocation granularity), i.e. 384 * 168 = 64512 in total. The
// producer/MMA warpgroup drops to 96 and the two softmax warpgroups rise to 200
// (128 * 96 + 256 * 200 = 63488), the split at which no d = 128 variant spills (88 / 208 left 16-byte spills in the control warps: 1-2 % slower).
// The build checks that ptxas launches this kernel at exactly kRegsLaunch.
constexpr int kRegsLaunch = 168;
constexpr int kRegsControl = 96;
constexpr int kRegsSoftmax = 200;
static_assert(128 * kRegsControl + 256 * kRegsSoftmax <= kThreads * kRegsLaunch, "register split");
// The block-sparse variant's walks over the mask bits, and the dense d = 64
// variant's separate S and P schedule, need more registers in the
// producer/MMA(/mask) warpgroup: 128 * 104 + 256 * 200 = 64512.
constexpr int kRegsControlSparse = 104;
constexpr int kRegsSoftmaxSparse = 200;
static_assert(128 * kRegsControlSparse + 256 * kRegsSoftmaxSparse <= kThreads * kRegsLaunch, "register split");
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kDrainLimitNs = 200000000ull;  // 0.2 s per drain wait
constexpr float kLazyRescaleLog2 = 8.0f;          // keep m while new scores exceed it by <= 2^8

// Block-mask ring (block-sparse variant): warp 2 reads the two mask rows of
// each item into bit words (bit j of row t: tile t keeps K/V block j, already
// clipped to the blocks the tile visits), with the kept-block counts and the
// highest and lowest blocks either tile keeps. Producer, MMA issuer and softmax warps walk
// the bits from shared memory, so no mask load sits on their paths.
constexpr int kMaskSlots = 3;  // three, so that the epilogue's staging slots fit beside the ring
constexpr int kMaskWords = 64;                        // up to 2048 blocks per row
constexpr int kMaskSlotBytes = 2 * kMaskWords * 4 + 16;
constexpr int kMaskConsumers = 1 + 1 + 8;             // producer, MMA issuer, 8 softmax warps
static_assert(kMaskWords * 32 == kSparseMaxBlocks, "mask ring size");

// barrier slots (KvFull / KvEmpty: one pair per K/V ring slot, which holds the K tile
// and the V tile of one step; room for up to kKvSlotsMax slots; MaskFull / MaskEmpty:
// room for up to kMaskSlotsMax block-mask slots)
constexpr int kKvSlotsMax = 3;
constexpr int kMaskSlotsMax = 4;
static_assert(kMaskSlots <= kMaskSlotsMax, "mask ring barriers");
enum : int {
  kBarQFull = 0, kBarQEmpty = 1, kBarKvFull = 2, kBarKvEmpty = 2 + kKvSlotsMax,
  kBarSFull = 2 + 2 * kKvSlotsMax, kBarPFull = kBarSFull + 2, kBarOFull = kBarPFull + 2, kBarMmaDone = kBarOFull + 2,
  kBarMaskFull = kBarMmaDone + 1, kBarMaskEmpty = kBarMaskFull + kMaskSlotsMax,
  // separate P buffers (dense d = 64): S_t read by the softmax, O_t += P_t V completed
  kBarSFree = kBarMaskFull + 2 * kMaskSlotsMax, kBarPvDone = kBarSFree + 2, kBarCount = kBarPvDone + 2
};

enum : int { kModeDense = 0, kModeSparse = 1, kModePaged = 2, kModeMasked = 3, kModeFp8 = 4 };

template <int D, int kMode>
struct TcLayout {
  static constexpr bool kFp8 = kMode == kModeFp8;
  // S_t(j + 1) issued as soon as the softmax has read S_t(j), not after P_t(j) V, where P
  // does not overwrite S: the dense, paged and masked variants at d = 64 (S_A, S_B, O_A and O_B take 384 TMEM
  // columns, so P_A and P_B get buffers of their own in the other 128, bf16 pairs, 64
  // columns each) and the FP8 variant (P in shared memory).
  static constexpr bool kPTmem = (kMode == kModeDense || kMode == kModePaged || kMode == kModeMasked) && D == 64;
  static constexpr bool kEarly = kPTmem || kFp8;
  static constexpr int kElem = kFp8 ? 1 : 2;      // bytes per Q/K/V element (E4M3 or bf16)
  static constexpr int kQBytes = BM * D * kElem;  // one Q tile
  static constexpr int kKVBytes = BN * D * kElem;
  // K/V ring slots: three for FP8 (its tiles take half the room), two elsewhere
  static constexpr int kStages = kFp8 ? 3 : 2;
  static_assert(kStages <= kKvSlotsMax, "K/V ring barriers");
  static constexpr int kOffQ = 0;                 // Q_A then Q_B
  static constexpr int kOffK = kOffQ + 2 * kQBytes;
  static constexpr int kOffV = kOffK + kStages * kKVBytes;
  // Epilogue staging: each softmax warp writes its 32 rows of one 64-column half of O (bf16,
  // 128-byte swizzle) into a 4 KB slot of its own and stores them with one TMA box.
  static constexpr int kStageSlot = 32 * 128;
  static constexpr int kOffStage = kOffV + kStages * kKVBytes;
  static constexpr int kOffBar = kOffStage + 8 * kStageSlot;
  static constexpr int kNumBars = kEarly ? kBarCount : kBarSFree;
  static constexpr int kBarStall = kNumBars;      // test hook: a barrier no role arrives on
  static constexpr int kOffHolder = kOffBar + (kNumBars + 1) * 8;
  static constexpr int kOffAbort = kOffHolder + 8;
  static constexpr int kOffMask = kOffAbort + 8;  // block-mask ring (block-sparse variant)
  // FP8 variant: P_A, P_B as E4M3 128 x 128 tiles in shared memory (128-byte swizzle)
  static constexpr int kOffP = (kOffMask + (kMode == kModeSparse ? kMaskSlots * kMaskSlotBytes : 0) + 1023) / 1024 * 1024;
  static constexpr int kPBytes = kFp8 ? BM * BN : 0;
  // + slack to align the base to 1024 B; at least 117 KB so that a second CTA
  // (which would block in tcgen05.alloc) never shares the SM
  static constexpr int kUsed = kOffP + 2 * kPBytes + 1024;
  static constexpr int kBytes = kUsed > 117 * 1024 ? kUsed : 117 * 1024;
  static_assert(kBytes <= 227 * 1024, "shared memory");
  // TMEM columns: fp32 scores S_A, S_B (bf16 variants: P_X in bf16 over their first 64
  // columns), fp32 O_A, O_B.
  __host__ __device__ static constexpr uint32_t col_s(int t) { return t ? 128u : 0u; }
  __host__ __device__ static constexpr uint32_t col_o(int t) { return t ? 256u + D : 256u; }
  __host__ __device__ static constexpr uint32_t col_p(int t) { return t ? 448u : 384u; }  // kPTmem only
  static_assert(256 + 2 * D <= kTmemCols, "TMEM budget");
  static_assert(!kPTmem || 256 + 2 * D <= 384, "TMEM budget with P buffers");
};

struct Item {
  int b, h, base, row0, L;  // L: query rows of the sequence (its length, or the chunk's)
  int Lk, off;              // keys of the sequence; query i sees keys j <= i + off if causal
  int n[2];   // K/V tiles tile A / tile B must visit (0: tile B has no row of the sequence)
  bool valid;
};

// Work-item order. Heads (b, h) are taken in groups whose items fill about four
// rounds of the grid when a head has at least 32 query-tile pairs, else two
// (measured against one to sixteen rounds: four is 6 % faster than two on
// 32k-token causal sequences, the same on 4k-token ones, and 20 % slower on the
// short packed sequences of a varlen batch), and with at least 32 pairs a group
// takes the heads of up to 8 KV heads if that is more (each KV head's K/V is then
// streamed by many CTAs at once and the group's items balance better over the grid:
// causal GQA B=1 Hq=32 Hkv=8 N=32768 6.51 -> 6.35 ms, B=2 N=16384 3.42 -> 3.36 ms,
// MHA B=1 H=32 N=32768 6.98 -> 6.56 ms); inside a group the items go heaviest causal Q pair first
// (all heads of the group at one pair index, then the next), and the grid walks
// the item list in alternating direction round by round ("snake"), so each CTA
// pairs heavy items with light ones while the K/V of the few heads in flight
// stay in L2.
struct Schedule {
  int pairs, heads, group, total;
};

__device__ __forceinline__ Schedule make_schedule(const PrefillParams& p) {
  Schedule s;
  s.pairs = (p.N + kRowsPerItem - 1) / kRowsPerItem;
  s.heads = p.B * p.Hq;
  const int G = p.Hq / p.Hkv;
  const int rounds = s.pairs >= 32 ? 4 : 2;                 // grid rounds per group
  int grp = (rounds * (int)gridDim.x + s.pairs - 1) / s.pairs;  // heads per group
  if (s.pairs >= 32) grp = max(grp, 8 * G);                 // long sequences: up to 8 KV heads at once
  grp = ((grp + G - 1) / G) * G;                            // whole GQA groups
  s.group = grp < s.heads ? grp : s.heads;
  s.total = s.heads * s.pairs;
  return s;
}

// k-th item of this CTA, or -1 past the end.
__device__ __forceinline__ int item_index(const Schedule& s, int k) {
  const int G = (int)gridDim.x;
  const int idx = k * G + ((k & 1) ? (G - 1 - (int)blockIdx.x) : (int)blockIdx.x);
  return idx < s.total ? idx : -1;
}

__device__ __forceinline__ Item decode_item(const PrefillParams& p, const Schedule& s, int it) {
  Item x;
  const int per_group = s.group * s.pairs;
  const int g = it / per_group;
  const int rem = it - g * per_group;
  const int gh = min(s.group, s.heads - g * s.group);       // heads in this (maybe last) group
  const int rank = rem / gh;
  const int bh = g * s.group + (rem - rank * gh);
  const int pair = s.pairs - 1 - rank;
  x.b = bh / p.Hq;
  x.h = bh - x.b * p.Hq;
  x.base = pair * kRowsPerItem;
  if (p.cu_seqlens) {
    const int start = __ldg(p.cu_seqlens + x.b);
    const int end = __ldg(p.cu_seqlens + x.b + 1);
    // paged: the chunk's queries are the last L of the sequence's Lk context tokens
    const int lk = p.seqlens_k ? __ldg(p.seqlens_k + x.b) : end - start;
    if (start < 0 || end < start || end > p.total_rows || end - start > p.N ||
        (p.seqlens_k && (lk < end - start || lk > p.max_pages * p.page_size))) {
      x.valid = false;
      x.row0 = x.L = x.Lk = x.off = x.n[0] = x.n[1] = 0;
      if (pair == 0 && x.h == 0 && (threadIdx.x & 31) == 0) record_status(p.status, kStatusDeviceCheck);
      return x;
    }
    x.row0 = start;
    x.L = end - start;
    x.Lk = lk;
  } else {
    x.row0 = x.b * p.N;
    x.L = x.Lk = p.N;
  }
  x.off = x.Lk - x.L;
  x.valid = x.base < x.L;
  const int kv_tiles = (x.Lk + BN - 1) / BN;
  const bool has_b = x.base + BM < x.L;
  if (p.causal) {  // up to the key the tile's last row sees
    x.n[0] = min((min(x.base + BM, x.L) - 1 + x.off) / BN + 1, kv_tiles);
    x.n[1] = has_b ? min((min(x.base + 2 * BM, x.L) - 1 + x.off) / BN + 1, kv_tiles) : 0;
  } else {
    x.n[0] = kv_tiles;
    x.n[1] = has_b ? kv_tiles : 0;
  }
  return x;
}

// Walks the kept blocks of one mask row (sel = 1 << t) or of the union of both
// rows (sel = 3) in decreasing order (the diagonal block first under the causal
// rule, as the dense variants visit their key tiles). The current word of each row
// is held in registers, so a step costs a count-leading-zeros; shared memory is
// read once per 32 blocks. Bits past a row's n[t] are zero.
struct BitWalk {
  const uint32_t* w;
  int sel, wi, bit;
  uint32_t u0, u1, rem;
  __device__ __forceinline__ BitWalk(const uint32_t* words, int sel_, int end)
      : w(words), sel(sel_), wi((end + 31) >> 5), bit(0), u0(0), u1(0), rem(0) {}
  __device__ __forceinline__ int next() {  // next kept block, or -1
    while (rem == 0) {
      if (--wi < 0) return -1;
      u0 = (sel & 1) ? w[wi] : 0u;
      u1 = (sel & 2) ? w[kMaskWords + wi] : 0u;
      rem = u0 | u1;
    }
    bit = 31 - __clz(rem);
    rem &= ~(1u << bit);
    return wi * 32 + bit;
  }
  __device__ __forceinline__ bool kept(int t) const { return ((t ? u1 : u0) >> bit) & 1u; }
};

// Drain wait: bounded, ignores the abort flag (used on the way out).
__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kDrainLimitNs) break;
  }
}

// Warp-uniform wait: lane 0 polls, the verdict is broadcast so that every
// lane takes the same path into the warp-collective tcgen05.ld/st.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort, int* status,
                                          uint64_t limit_ns) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort, status, limit_ns);
  ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  return ok;
}

// Variants of the kernel (template argument kMode).

template <int D, int kMode>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                      const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap to,
                      const PrefillParams p) {
  constexpr bool kSparse = kMode == kModeSparse;  // fixed block mask, zero blocks skipped
  constexpr bool kPaged = kMode == kModePaged;    // K/V through a block table
  constexpr bool kMasked = kMode == kModeMasked;  // additive bf16 mask M on the scores
  constexpr bool kFp8 = kMode == kModeFp8;        // E4M3 Q, K, V; P in E4M3 through shared memory
  // key tiles visited from the last (the diagonal under the causal rule) down to 0, so that the
  // two tiles of an item finish together (block-sparse: the bit walks go down likewise)
  constexpr bool kReverse = !kSparse;
  static_assert(!kFp8 || D == 128, "FP8 tiles are 128 one-byte columns: one 128-byte swizzle span");
  constexpr int kChunks = kFp8 ? 1 : D / 64;      // 128-byte boxes per tile row
  using Lay = TcLayout<D, kMode>;
  constexpr bool kEarly = Lay::kEarly;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sb + Lay::kOffBar + 8 * i; };
  volatile int* abort = reinterpret_cast<volatile int*>(smem + Lay::kOffAbort);
  // u-th item's block-mask slot: bit words of rows 0 and 1, then {cnt0, cnt1, last}
  auto mask_slot = [&](uint32_t u) -> const uint32_t* {
    return reinterpret_cast<const uint32_t*>(smem + Lay::kOffMask + (u % kMaskSlots) * kMaskSlotBytes);
  };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < Lay::kNumBars; ++i)
      mbar_init(bar(i), (i == kBarPFull || i == kBarPFull + 1 || i == kBarSFree || i == kBarSFree + 1) ? 4
                        : (i >= kBarMaskEmpty && i < kBarMaskEmpty + kMaskSlots)                ? kMaskConsumers
                                                                                                 : 1);
    mbar_init(bar(Lay::kBarStall), 1);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tq);
    tma_prefetch_desc(&tk);
    tma_prefetch_desc(&tv);
    tma_prefetch_desc(&to);
  }
  if (warp == 1) {
    tmem_alloc(sb + Lay::kOffHolder, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + Lay::kOffHolder);

  const Schedule sch = make_schedule(p);
  const int G = p.Hq / p.Hkv;

  if (warp < 4) {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"((kSparse || Lay::kPTmem) ? kRegsControlSparse : kRegsControl));
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Lane 0 issues every copy; the paged variant runs lanes 0-7 through the same
    // loop (each lane waits on the same barriers) and lane i copies page i of a tile,
    // because one thread issuing a tile's 2 x (128 / page_size) boxes in sequence
    // cannot keep up with the tensor core for small pages.
    const bool leader = lane == 0;
    if (kPaged ? lane < BN / 16 : leader) {
      uint32_t nq = 0, nk = 0, nm = 0;  // nk: K/V ring steps
      const uint64_t pol_q = policy_evict_first(), pol_kv = policy_evict_last();
      for (int k = 0;; ++k) {
        const int it = item_index(sch, k);
        if (it < 0) break;
        const Item x = decode_item(p, sch, it);
        if (!x.valid) continue;
        const int hkv = x.h / G;
        const int n = max(x.n[0], x.n[1]);
        const uint32_t* mw = nullptr;
        if constexpr (kSparse) {
          if (!mbar_wait(bar(kBarMaskFull + nm % kMaskSlots), (nm / kMaskSlots) & 1, abort, p.status, p.wait_ns))
            break;
          mw = mask_slot(nm);
          if ((int)mw[2 * kMaskWords + 2] < 0) {  // neither tile keeps a block: Q is not needed
            mbar_arrive(bar(kBarMaskEmpty + nm % kMaskSlots));
            ++nm;
            continue;
          }
        }
        if (!mbar_wait(bar(kBarQEmpty), (nq & 1) ^ 1, abort, p.status, p.wait_ns)) break;
        if (leader) {
          mbar_arrive_expect_tx(bar(kBarQFull), 2 * Lay::kQBytes);
#pragma unroll
          for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int dc = 0; dc < kChunks; ++dc)
              tma_load_3d(sb + Lay::kOffQ + t * Lay::kQBytes + dc * BM * 128, &tq, bar(kBarQFull), dc * 64, x.h,
                          x.row0 + x.base + t * BM, pol_q);
        }
        ++nq;
        // K or V tile j (keys [128 j, 128 j + 128)) into one ring stage. Paged: one box
        // of page_size rows per page, at the page's rows of the pool (read through the
        // block table, each entry checked); slots past the sequence's last page read a
        // box beyond the pool, which the copy fills with zeros. The boxes stack into the
        // same swizzled layout as one 128-row box (page_size is a multiple of 8 rows).
        auto issue_kv = [&](const CUtensorMap* map, uint32_t dst, uint32_t full, int j, bool is_v) {
          (void)is_v;
          if constexpr (kPaged) {
            const int P = p.page_size, per = BN / P;  // per <= 8 (page_size >= 16)
            const int i = lane;                       // this lane's page of the tile
            if (i < per) {
              const int slot = j * per + i;
              int prow = p.num_pages * P;
              if (slot < (x.Lk + P - 1) / P) {
                const int pg = __ldg(p.block_table + (size_t)x.b * p.max_pages + slot);
                if (pg >= 0 && pg < p.num_pages)
                  prow = pg * P;
                else
                  record_status(p.status, kStatusDeviceCheck);
              }
#pragma unroll
              for (int dc = 0; dc < D / 64; ++dc)
                tma_load_3d(dst + dc * BN * 128 + i * P * 128, map, full, dc * 64, hkv, prow, pol_kv);
            }
          } else {
#pragma unroll
            for (int dc = 0; dc < kChunks; ++dc)
              tma_load_3d(dst + dc * BN * 128, map, full, dc * 64, hkv, x.row0 + j * BN, pol_kv);
          }
        };
        // in the order the MMA warp consumes them, one ring slot per step: K0; K1 V0;
        // K2 V1; ...; V(last) (over the blocks either tile visits)
        bool ok = true;
        if constexpr (kSparse) {
          int prev = -1;
          // the same steps over the union of the blocks either tile keeps: K of this block
          // and V of the previous kept one, then V of the last one alone
          BitWalk walk(mw, 3, n);
          for (int j = walk.next(); ok; j = walk.next()) {
            const uint32_t st = nk % Lay::kStages;
            if (!mbar_wait(bar(kBarKvEmpty + st), ((nk / Lay::kStages) & 1) ^ 1, abort, p.status, p.wait_ns)) {
              ok = false;
              break;
            }
            if (leader) mbar_arrive_expect_tx(bar(kBarKvFull + st), ((j >= 0) + (prev >= 0)) * Lay::kKVBytes);
            if (j >= 0) issue_kv(&tk, sb + Lay::kOffK + st * Lay::kKVBytes, bar(kBarKvFull + st), j, false);
            if (prev >= 0) issue_kv(&tv, sb + Lay::kOffV + st * Lay::kKVBytes, bar(kBarKvFull + st), prev, true);
            ++nk;
            if (j < 0) break;
            prev = j;
          }
          mbar_arrive(bar(kBarMaskEmpty + nm % kMaskSlots));
          ++nm;
        } else {
          // step s: K_s (s < n) and V_{s-1} (s > 0) into slot nk mod 2 of both rings, under
          // one full / empty barrier pair (step 0 carries K_0 alone, step n V_{n-1} alone):
          // the MMA issuer takes them in the same step, so it saves a wait and a commit per
          // step, which the tensor core would otherwise wait out (against separate K and V
          // barriers: causal MHA 0.485 -> 0.479 ms, varlen d = 64 0.127 -> 0.119 ms)
          for (int s = 0; ok && s <= n; ++s) {
            const uint32_t st = nk % Lay::kStages;
            if (!mbar_wait(bar(kBarKvEmpty + st), ((nk / Lay::kStages) & 1) ^ 1, abort, p.status, p.wait_ns)) {
              ok = false;
              break;
            }
            if (leader) mbar_arrive_expect_tx(bar(kBarKvFull + st), ((s < n) + (s > 0)) * Lay::kKVBytes);
            if (s < n) issue_kv(&tk, sb + Lay::kOffK + st * Lay::kKVBytes, bar(kBarKvFull + st), kReverse ? n - 1 - s : s, false);
            if (s > 0) issue_kv(&tv, sb + Lay::kOffV + st * Lay::kKVBytes, bar(kBarKvFull + st), kReverse ? n - s : s - 1, true);
            ++nk;
          }
        }
        if (!ok) break;
      }
      // no copy may land after the CTA is gone: wait for the last armed phase of each barrier
      if (nq) mbar_drain(bar(kBarQFull), (nq - 1) & 1);
      for (uint32_t st = 0; st < (uint32_t)Lay::kStages; ++st) {
        const uint32_t c = nk > st ? (nk - st + Lay::kStages - 1) / Lay::kStages : 0;  // steps loaded into slot st
        if (c) mbar_drain(bar(kBarKvFull + st), (c - 1) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(BM, BN, 0);  // Q K^T: both K-major
      constexpr uint32_t idO = idesc_bf16_f32(BM, D, 1);   // P V: V is MN-major (d contiguous)
      uint32_t nq = 0, nk = 0;                             // nk: K/V ring steps consumed
      uint32_t np[2] = {0, 0};                             // P_X buffers consumed so far
      uint32_t si[2] = {0, 0};                             // S_X issued (dense d = 64)
      // Descriptor bases, built once. The start-address field (bits 0-13, in
      // 16-byte units) of each per-MMA descriptor is the base plus a
      // compile-time offset, so issuing an MMA costs no descriptor arithmetic.
      const uint64_t qd0 = smem_desc_sw128(sb + Lay::kOffQ, 16, 1024);
      const uint64_t qd1 = smem_desc_sw128(sb + Lay::kOffQ + Lay::kQBytes, 16, 1024);
      // ring slot st: with two slots one of two descriptors; with three, the slot-0
      // descriptor plus st tiles (the start address field counts 16-byte units; every
      // slot lies below 256 KB, so it never overflows)
      const uint64_t kd0 = smem_desc_sw128(sb + Lay::kOffK, 16, 1024);
      const uint64_t kd1 = smem_desc_sw128(sb + Lay::kOffK + Lay::kKVBytes, 16, 1024);
      // V: MN-major (d contiguous, 128-byte column blocks BN * 128 bytes apart; the FP8
      // tile's d = 128 bytes is a single block)
      const uint64_t vd0 = smem_desc_sw128(sb + Lay::kOffV, BN * 128, 1024);
      const uint64_t vd1 = smem_desc_sw128(sb + Lay::kOffV + Lay::kKVBytes, BN * 128, 1024);
      auto slot_desc = [&](uint64_t d0, uint64_t d1, uint32_t st) -> uint64_t {
        if constexpr (Lay::kStages == 2)
          return st ? d1 : d0;
        else
          return d0 + (uint64_t)(st * (Lay::kKVBytes >> 4));
      };
      auto issue_s = [&](int t, uint32_t kst) {
        const uint32_t d_tmem = tmem + Lay::col_s(t);
        const uint64_t a0 = t ? qd1 : qd0, b0 = slot_desc(kd0, kd1, kst);
        if constexpr (kFp8) {  // K = 32 one-byte elements (32 bytes) per instruction
          constexpr uint32_t idS8 = idesc_e4m3_f32(BM, BN, 0);
          mma_ss_e4m3<false>(d_tmem, a0, b0, idS8);
#pragma unroll
          for (int ks = 1; ks < D / 32; ++ks) mma_ss_e4m3<true>(d_tmem, a0 + (uint64_t)(ks * 2), b0 + (uint64_t)(ks * 2), idS8);
          mma_commit(bar(kBarSFull + t));
          return;
        }
        mma_ss_c<false>(d_tmem, a0, b0, idS);
#pragma unroll
        for (int ks = 1; ks < D / 16; ++ks) {
          constexpr int kAtomQ = BM * 128 / 16, kAtomK = BN * 128 / 16;  // 16-byte units per swizzle atom column
          mma_ss_c<true>(d_tmem, a0 + (uint64_t)((ks >> 2) * kAtomQ + (ks & 3) * 2),
                         b0 + (uint64_t)((ks >> 2) * kAtomK + (ks & 3) * 2), idS);
        }
        mma_commit(bar(kBarSFull + t));
      };
      auto issue_pv = [&](int t, uint32_t vst, bool acc) -> bool {
        if (!mbar_wait(bar(kBarPFull + t), np[t] & 1, abort, p.status, p.wait_ns)) return false;
        ++np[t];
        tc_fence_after();
        const uint32_t p_tmem = tmem + (Lay::kPTmem ? Lay::col_p(t) : Lay::col_s(t)), o_tmem = tmem + Lay::col_o(t);
        const uint64_t b0 = slot_desc(vd0, vd1, vst);
        if constexpr (kFp8) {  // O += P V with P (E4M3, shared memory, K-major) and V (MN-major)
          constexpr uint32_t idO8 = idesc_e4m3_f32(BM, D, 1);
          const uint64_t a0 = smem_desc_sw128(sb + Lay::kOffP + t * Lay::kPBytes, 16, 1024);
          mma_ss_e4m3_p(o_tmem, a0, b0, idO8, acc ? 1u : 0u);
          // K = 32 keys per instruction: P advances 32 bytes along its rows, V 32 rows of 128 bytes
#pragma unroll
          for (int ks = 1; ks < BN / 32; ++ks)
            mma_ss_e4m3<true>(o_tmem, a0 + (uint64_t)(ks * 2), b0 + (uint64_t)(ks * 32 * 128 / 16), idO8);
          return true;
        }
        mma_ts(o_tmem, p_tmem, b0, idO, acc ? 1u : 0u);
#pragma unroll
        for (int ks = 1; ks < BN / 16; ++ks) mma_ts_acc(o_tmem, p_tmem + ks * 8, b0 + (uint64_t)(ks * 16 * 128 / 16), idO);
        return true;
      };
      bool ok = true;
      uint32_t nm = 0;
      for (int k = 0; ok; ++k) {
        const int it = item_index(sch, k);
        if (it < 0) break;
        const Item x = decode_item(p, sch, it);
        if (!x.valid) continue;
        if constexpr (kSparse) {
          // walk the blocks either tile keeps: per block j, O_t += P_t(prev) V_prev for each tile
          // that kept the previous block, then S_t = Q_t K_j^T for each tile that keeps j
          if (!mbar_wait(bar(kBarMaskFull + nm % kMaskSlots), (nm / kMaskSlots) & 1, abort, p.status, p.wait_ns))
            break;
          const uint32_t* mw = mask_slot(nm);
          const int cnt[2] = {(int)mw[2 * kMaskWords], (int)mw[2 * kMaskWords + 1]};
          const int last = (int)mw[2 * kMaskWords + 2], low = (int)mw[2 * kMaskWords + 3];
          if (last < 0) {  // the producer loads no Q for this item
            mbar_arrive(bar(kBarMaskEmpty + nm % kMaskSlots));
            ++nm;
            continue;
          }
          if (!mbar_wait(bar(kBarQFull), nq & 1, abort, p.status, p.wait_ns)) break;
          ++nq;
          tc_fence_after();
          const int n = max(x.n[0], x.n[1]);
          int done0 = 0, done1 = 0;          // P V products issued per tile
          bool had0 = false, had1 = false;    // tile kept the previous union block
          BitWalk walk(mw, 3, n);
          for (int j = walk.next(); j >= 0; j = walk.next()) {
            const bool a0 = walk.kept(0), a1 = walk.kept(1);
            const uint32_t kst = nk % Lay::kStages, vst = kst;  // K of block j, V of the previous kept block
            if (!mbar_wait(bar(kBarKvFull + kst), (nk / Lay::kStages) & 1, abort, p.status, p.wait_ns)) {
              ok = false;
              break;
            }
            tc_fence_after();
            if (had0) {
              if (!issue_pv(0, vst, done0 > 0)) { ok = false; break; }
              if (++done0 == cnt[0]) mma_commit(bar(kBarOFull + 0));
            }
            if (a0) issue_s(0, kst);
            if (had1) {
              if (!issue_pv(1, vst, done1 > 0)) { ok = false; break; }
              if (++done1 == cnt[1]) mma_commit(bar(kBarOFull + 1));
            }
            if (a1) issue_s(1, kst);
            had0 = a0;
            had1 = a1;
            mma_commit(bar(kBarKvEmpty + kst));
            ++nk;
            if (j == low) mma_commit(bar(kBarQEmpty));  // the walk's last block
          }
          if (!ok) break;
          const uint32_t vst = nk % Lay::kStages;  // V of the last kept block alone
          if (!mbar_wait(bar(kBarKvFull + vst), (nk / Lay::kStages) & 1, abort, p.status, p.wait_ns)) break;
          tc_fence_after();
          if (had0) {
            if (!issue_pv(0, vst, done0 > 0)) break;
            mma_commit(bar(kBarOFull + 0));
          }
          if (had1) {
            if (!issue_pv(1, vst, done1 > 0)) break;
            mma_commit(bar(kBarOFull + 1));
          }
          mma_commit(bar(kBarKvEmpty + vst));
          ++nk;
          mbar_arrive(bar(kBarMaskEmpty + nm % kMaskSlots));
          ++nm;
          continue;
        }
        const int nA = x.n[0], nB = x.n[1];
        const int n = max(nA, nB);
        // tile t takes part in steps [f_t, f_t + n_t) (reverse order: the last n_t steps)
        const int fA = kReverse ? n - nA : 0, fB = kReverse ? n - nB : 0;
        auto in_a = [&](int s) { return s >= fA && s < fA + nA; };
        auto in_b = [&](int s) { return s >= fB && s < fB + nB; };
        if (!mbar_wait(bar(kBarQFull), nq & 1, abort, p.status, p.wait_ns)) break;
        ++nq;
        tc_fence_after();
        if constexpr (kEarly) {
          // per K/V tile j: S_A(j) and S_B(j) once each softmax has read its previous S,
          // then O_t += P_t(j-1) V_{j-1} once P_t(j-1) is written
          auto early_s = [&](int t, uint32_t kst) -> bool {
            if (si[t] > 0 && !mbar_wait(bar(kBarSFree + t), (si[t] - 1) & 1, abort, p.status, p.wait_ns))
              return false;
            ++si[t];
            tc_fence_after();
            issue_s(t, kst);
            return true;
          };
          auto early_pv = [&](int t, uint32_t vst, bool acc) -> bool {
            if (!issue_pv(t, vst, acc)) return false;
            mma_commit(bar(kBarPvDone + t));  // P_t's buffer is free and O_t holds the tile
            return true;
          };
          for (int j = 0; ok && j <= n; ++j) {
            // step j: S_A(j), S_B(j) (j < n) and O_t += P_t(j-1) V_{j-1} (j > 0), K_j and
            // V_{j-1} in slot nk mod 2 under one barrier pair
            const uint32_t st = nk % Lay::kStages;
            if (!mbar_wait(bar(kBarKvFull + st), (nk / Lay::kStages) & 1, abort, p.status, p.wait_ns) ||
                (in_a(j) && !early_s(0, st)) || (in_b(j) && !early_s(1, st))) {
              ok = false;
              break;
            }
            if (j == n - 1) mma_commit(bar(kBarQEmpty));
            if (j > 0) {
              tc_fence_after();
              if ((in_a(j - 1) && !early_pv(0, st, j - 1 > fA)) || (in_b(j - 1) && !early_pv(1, st, j - 1 > fB))) {
                ok = false;
                break;
              }
            }
            mma_commit(bar(kBarKvEmpty + st));
            ++nk;
          }
          continue;
        }
        // j = 0
        {
          const uint32_t kst = nk % Lay::kStages;
          if (!mbar_wait(bar(kBarKvFull + kst), (nk / Lay::kStages) & 1, abort, p.status, p.wait_ns)) break;
          tc_fence_after();
          if (in_a(0)) issue_s(0, kst);
          if (in_b(0)) issue_s(1, kst);
          mma_commit(bar(kBarKvEmpty + kst));
          ++nk;
          if (n == 1) mma_commit(bar(kBarQEmpty));
        }
        for (int j = 1; ok && j < n; ++j) {
          const uint32_t kst = nk % Lay::kStages, vst = kst;  // K_j and V_{j-1}: one slot, one barrier
          if (!mbar_wait(bar(kBarKvFull + kst), (nk / Lay::kStages) & 1, abort, p.status, p.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (in_a(j - 1)) {
            if (!issue_pv(0, vst, j - 1 > fA)) { ok = false; break; }
            if (j - 1 == fA + nA - 1) mma_commit(bar(kBarOFull + 0));
          }
          if (in_a(j)) issue_s(0, kst);
          if (in_b(j - 1)) {
            if (!issue_pv(1, vst, j - 1 > fB)) { ok = false; break; }
            if (j - 1 == fB + nB - 1) mma_commit(bar(kBarOFull + 1));
          }
          if (in_b(j)) issue_s(1, kst);
          mma_commit(bar(kBarKvEmpty + kst));
          ++nk;
          if (j == n - 1) mma_commit(bar(kBarQEmpty));
        }
        if (!ok) break;
        // tail: the last P V of each tile
        {
          const uint32_t vst = nk % Lay::kStages;  // V_{n-1} alone in the item's last slot
          if (!mbar_wait(bar(kBarKvFull + vst), (nk / Lay::kStages) & 1, abort, p.status, p.wait_ns)) break;
          tc_fence_after();
          if (in_a(n - 1)) {
            if (!issue_pv(0, vst, n - 1 > fA)) break;
            mma_commit(bar(kBarOFull + 0));
          }
          if (in_b(n - 1)) {
            if (!issue_pv(1, vst, n - 1 > fB)) break;
            mma_commit(bar(kBarOFull + 1));
          }
          mma_commit(bar(kBarKvEmpty + vst));
          ++nk;
        }
      }
      // every MMA (and every commit before this one) has landed before TMEM is freed
      mma_commit(bar(kBarMmaDone));
      mbar_drain(bar(kBarMmaDone), 0);
    }
  } else if (kSparse && warp == 2) {
    // ------------------------------------------------------------ block-mask reader
    // Per item: lane i tests blocks 32 w + i of both mask rows, a ballot packs
    // them into word w; blocks at or past n[t] (causal skip, sequence end) are 0.
    const int nb = (p.N + BN - 1) / BN;
    uint32_t nm = 0;
    for (int k = 0;; ++k) {
      const int it = item_index(sch, k);
      if (it < 0) break;
      const Item x = decode_item(p, sch, it);
      if (!x.valid) continue;
      if (!warp_wait(bar(kBarMaskEmpty + nm % kMaskSlots), ((nm / kMaskSlots) & 1) ^ 1, abort, p.status, p.wait_ns)) break;
      uint32_t* w = reinterpret_cast<uint32_t*>(smem + Lay::kOffMask + (nm % kMaskSlots) * kMaskSlotBytes);
      const int nw = (max(x.n[0], x.n[1]) + 31) >> 5;   // <= kMaskWords: nb <= kSparseMaxBlocks
      int cnt[2] = {0, 0}, last = -1, low = 1 << 30;
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const uint8_t* mrow = p.block_mask + ((size_t)(x.h % p.mask_heads) * nb + (x.base / BM + t)) * nb;
        for (int w0 = 0; w0 < nw; w0 += 4) {
          uint32_t v[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int j = (w0 + i) * 32 + lane;
            v[i] = j < x.n[t] ? __ldg(mrow + j) : 0u;      // j < n[t] <= nb: inside row t
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t bits = __ballot_sync(0xffffffffu, v[i] != 0u);
            if (w0 + i < nw) {
              if (lane == 0) w[t * kMaskWords + w0 + i] = bits;
              cnt[t] += __popc(bits);
              if (bits) {
                last = max(last, (w0 + i) * 32 + 31 - __clz(bits));
                low = min(low, (w0 + i) * 32 + __ffs(bits) - 1);
              }
            }
          }
        }
      }
      if (lane == 0) {
        w[2 * kMaskWords] = (uint32_t)cnt[0];
        w[2 * kMaskWords + 1] = (uint32_t)cnt[1];
        w[2 * kMaskWords + 2] = (uint32_t)last;
        w[2 * kMaskWords + 3] = (uint32_t)low;   // the walk's last block (it goes down)
        mbar_arrive(bar(kBarMaskFull + nm % kMaskSlots));  // release: the words above are visible
      }
      __syncwarp();
      ++nm;
    }
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"((kSparse || Lay::kPTmem) ? kRegsSoftmaxSparse : kRegsSoftmax));
    // ------------------------------------------------------------ softmax (tile t)
    const int t = (warp - 4) >> 2;           // 0: tile A (warps 4-7), 1: tile B (warps 8-11)
    const int q4 = warp & 3;                 // TMEM lane quarter this warp may touch
    const int r = q4 * 32 + lane;            // query row within the tile
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const uint32_t s_col = tmem + lane_off + Lay::col_s(t);
    const uint32_t o_col = tmem + lane_off + Lay::col_o(t);
    const float sl2 = p.scale * kLog2e;      // scores go to the log2 domain
    const bool neg = sl2 < 0.f;
    const uint64_t sl2x2 = f2_pack(sl2, sl2);
    const uint64_t scale2 = f2_pack(p.scale, p.scale);
    uint32_t ns = 0, no = 0;                 // S_t and O_t completions seen
    uint32_t npv = 0;                        // O_t += P_t V completions seen (dense d = 64)
    const uint32_t p_col = tmem + lane_off + (Lay::kPTmem ? Lay::col_p(t) : Lay::col_s(t));
    uint32_t nm = 0;                         // block-mask slots consumed
    // this warp's 4 KB staging slot (the epilogue's O stores; the masked variant's mask rows)
    uint8_t* slot = smem + Lay::kOffStage + (warp - 4) * Lay::kStageSlot;
    const uint32_t slot_s = sb + Lay::kOffStage + (warp - 4) * Lay::kStageSlot;
    bool slot_store = false;                 // an O store from the slot may still be reading it
    bool ok = true;
    // test hook: a wait that runs out (nothing arrives on the stall barrier), after which
    // every role stops, drains and frees TMEM; the outputs stay unwritten
    if (p.debug_stall && !warp_wait(bar(Lay::kBarStall), 0, abort, p.status, p.wait_ns)) ok = false;
    for (int k = 0; ok; ++k) {
      const int it = item_index(sch, k);
      if (it < 0) break;
      const Item x = decode_item(p, sch, it);
      if (!x.valid) continue;
      const uint32_t* mw = nullptr;
      // this tile's K/V tile count, selected rather than indexed (a run-time index into the
      // item's array would put the whole item in local memory)
      const int nt = t ? x.n[1] : x.n[0];
      int kept_blocks = nt;
      if constexpr (kSparse) {
        const uint32_t mb = bar(kBarMaskFull + nm % kMaskSlots), mp = (nm / kMaskSlots) & 1;
        if (!warp_wait(mb, mp, abort, p.status, p.wait_ns)) break;
        mbar_try_wait(mb, mp);  // completed: this lane's own acquire of the mask words
        mw = mask_slot(nm);
        kept_blocks = (int)mw[2 * kMaskWords + t];
      }
      // the mask words stay in use until every consumer of the slot releases it
      auto release_mask = [&]() {
        if constexpr (kSparse) {
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kBarMaskEmpty + nm % kMaskSlots));
          ++nm;
        }
      };
      if (nt == 0) {
        release_mask();
        continue;
      }
      const int row = x.base + t * BM + r;
      const int lim = p.causal ? min(row + x.off + 1, x.Lk) : x.Lk;  // keys < lim are visible
      if constexpr (kSparse) {  // a tile that keeps no block: O = 0, lse = -inf
        if (kept_blocks == 0) {
          release_mask();
          if (row < x.L) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.o) +
                                                  ((size_t)(x.row0 + row) * p.Hq + x.h) * D);
#pragma unroll
            for (int e = 0; e < D / 8; ++e) dst[e] = make_uint4(0, 0, 0, 0);
            if (p.lse) p.lse[((size_t)x.b * p.Hq + x.h) * p.N + row] = -CUDART_INF_F;
          }
          continue;
        }
      }
      float m = -CUDART_INF_F, l = 0.f;
      bool first = true;
      // additive mask: this row's entries (bf16), row clamped into the sequence (rows past it are not written)
      const __nv_bfloat16* mrow = nullptr;
      if constexpr (kMasked)
        mrow = static_cast<const __nv_bfloat16*>(p.mask) + (size_t)x.b * p.mask_sb + (size_t)x.h * p.mask_sh +
               (size_t)min(row, x.L - 1) * p.mask_ld;
      BitWalk walk(mw, 1 << t, nt);
      for (int j = kSparse ? walk.next() : (kReverse ? nt - 1 : 0); kSparse || kReverse ? j >= 0 : j < nt;
           j = kSparse ? walk.next() : (kReverse ? j - 1 : j + 1)) {
        // the tile's 128 mask entries, requested before waiting for S (16-byte loads
        // of whole 8-key groups; groups at or past the visible limit are not read)
        uint4 mv[kMasked ? BN / 16 : 1];
        auto load_mask = [&](int c8) {
          mv[c8] = j * BN + 8 * c8 < lim ? __ldg(reinterpret_cast<const uint4*>(mrow + j * BN + 8 * c8))
                                         : make_uint4(0u, 0u, 0u, 0u);
        };
        if constexpr (kMasked) {
          // the second half of the warp's 32 mask rows (keys 64-127 of the tile) goes to the
          // warp's staging slot by coalesced 16-byte copies (8 lanes per row, row rr at
          // 128 rr, chunk c at c ^ (rr mod 8); groups at or past the row's visible limit
          // are zero-filled without a read); the first half to registers, one row per thread
          __syncwarp();  // every lane has read the slot's previous contents
          if (slot_store) {  // an O store from the slot may still be reading it
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
            slot_store = false;
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int rr = 4 * i + (lane >> 3), cc = lane & 7;
            const int qrow = x.base + t * BM + q4 * 32 + rr;
            const int rlim = p.causal ? min(qrow + x.off + 1, x.Lk) : x.Lk;
            const int key0 = j * BN + BN / 2 + 8 * cc;
            const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(p.mask) + (size_t)x.b * p.mask_sb +
                                       (size_t)x.h * p.mask_sh + (size_t)min(qrow, x.L - 1) * p.mask_ld + key0;
            cp_async_16(slot_s + rr * 128 + ((cc ^ (rr & 7)) << 4), src, key0 < rlim ? 16u : 0u);
          }
          cp_async_commit();
          if (p.mask_v8) {  // 32-byte loads of whole 16-key groups (rows 32-byte aligned)
#pragma unroll
            for (int c16 = 0; c16 < BN / 32; ++c16) {
              if (j * BN + 16 * c16 < lim) {
                ldg_nc_32b(mrow + j * BN + 16 * c16, mv[2 * c16], mv[2 * c16 + 1]);
              } else {
                mv[2 * c16] = make_uint4(0u, 0u, 0u, 0u);
                mv[2 * c16 + 1] = make_uint4(0u, 0u, 0u, 0u);
              }
            }
          } else {
#pragma unroll
            for (int c8 = 0; c8 < BN / 16; ++c8) load_mask(c8);
          }
        }
        if (!warp_wait(bar(kBarSFull + t), ns & 1, abort, p.status, p.wait_ns)) {
          ok = false;
          break;
        }
        ++ns;
        tc_fence_after();
        float s[BN];
        const int kbase = j * BN;
        bool masked = kbase + BN > lim;  // causal diagonal tile or sequence end
        if constexpr (kMasked) {
          // masked scores s scale + M (natural-log units; log2(e) is applied with the
          // exponent), one packed FMA per column pair, 32 columns at a time so each
          // mask word dies as its scores arrive; keys past the visible limit -inf
          // (their p is 0 below)
          uint32_t u[BN];
          tmem_ld128(s_col, u);  // one wait for all 128 scores
          cp_async_wait_all();
          __syncwarp();  // the warp's copies of the second half have landed
#pragma unroll
          for (int q32 = 0; q32 < BN / 32; ++q32) {
            uint4 gq[4];  // this 32-column group's mask entries
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
              const int c8 = 4 * q32 + c4;
              gq[c4] = c8 < BN / 16 ? mv[c8 < BN / 16 ? c8 : 0]
                                    : *reinterpret_cast<const uint4*>(slot + lane * 128 + (((c8 - BN / 16) ^ (lane & 7)) << 4));
            }
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const int c = 32 * q32 + e;
              const uint4& g = gq[e >> 3];
              const uint32_t w = ((c & 7) >> 1) == 0 ? g.x : ((c & 7) >> 1) == 1 ? g.y : ((c & 7) >> 1) == 2 ? g.z : g.w;
              float t0, t1;
              f2_unpack(f2_fma(f2_pack(__uint_as_float(u[c]), __uint_as_float(u[c + 1])), scale2,
                               f2_pack(bf16_lo(w), bf16_hi(w))), t0, t1);
              s[c] = t0;
              s[c + 1] = t1;
            }
          }
          if constexpr (kEarly) {  // S_t(j) is in registers: the next product may overwrite it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarSFree + t));
          }
          if (masked) {
#pragma unroll
            for (int c = 0; c < BN; ++c)
              if (kbase + c >= lim) s[c] = -CUDART_INF_F;
          }
          masked = false;
        } else {
          {
            uint32_t u[BN];
            tmem_ld128(s_col, u);
#pragma unroll
            for (int e = 0; e < BN; ++e) s[e] = __uint_as_float(u[e]);
          }
          if constexpr (kEarly) {  // S_t(j) is in registers: the next product may overwrite it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarSFree + t));
          }
        }
        if (!kMasked && masked) {
#pragma unroll
          for (int c = 0; c < BN; ++c)
            if (kbase + c >= lim) s[c] = neg ? CUDART_INF_F : -CUDART_INF_F;
        }
        // row max (min for a negative scale): 8 independent chains of 3-input max
        float mx;
        {
          float a[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) a[i] = s[i];
          if (kMasked || !neg) {
#pragma unroll
            for (int c = 8; c < BN; c += 16)
#pragma unroll
              for (int i = 0; i < 8; ++i) a[i] = fmax3(a[i], s[c + i], s[c + 8 + i < BN ? c + 8 + i : c + i]);
            mx = fmax3(fmax3(a[0], a[1], a[2]), fmax3(a[3], a[4], a[5]), fmaxf(a[6], a[7]));
          } else {
#pragma unroll
            for (int c = 8; c < BN; c += 16)
#pragma unroll
              for (int i = 0; i < 8; ++i) a[i] = fmin3(a[i], s[c + i], s[c + 8 + i < BN ? c + 8 + i : c + i]);
            mx = fmin3(fmin3(a[0], a[1], a[2]), fmin3(a[3], a[4], a[5]), fminf(a[6], a[7]));
          }
        }
        const float m_cand = fmaxf(m, mx * (kMasked ? kLog2e : sl2));  // the masked scores carry the scale
        const bool need = m_cand > m + kLazyRescaleLog2;          // always true on the first tile
        const float m_new = __any_sync(0xffffffffu, need) ? m_cand : m;
        const float base = m_new == -CUDART_INF_F ? 0.f : m_new;
        const float alpha = ex2(m - base);                        // 1 when m is kept
        const uint64_t nbase2 = f2_pack(-base, -base);
        const uint64_t mul2 = kMasked ? f2_pack(kLog2e, kLog2e) : sl2x2;
        constexpr int kAcc = kMasked ? 2 : 8;  // packed row-sum partials (fewer registers when masked)
        uint64_t acc2[8] = {0ull, 0ull, 0ull, 0ull, 0ull, 0ull, 0ull, 0ull};  // row-sum partials, packed pairs
        // a column pair of P: bf16x2, or (FP8 variant) E4M3x2 in the low 16 bits
        auto pack_p = [](float p0, float p1) -> uint32_t {
          if constexpr (kFp8)
            return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(p0, p1), __NV_SATFINITE, __NV_E4M3);
          else
            return pack_bf16x2(p0, p1);
        };
        uint32_t pk[BN / 2];
        if (!masked) {
#pragma unroll
          for (int c = 0; c < BN; c += 2) {
            float a0, a1;
            f2_unpack(f2_fma(f2_pack(s[c], s[c + 1]), mul2, nbase2), a0, a1);
            const float p0 = ex2(a0), p1 = ex2(a1);
            acc2[(c >> 1) & (kAcc - 1)] = f2_add(acc2[(c >> 1) & (kAcc - 1)], f2_pack(p0, p1));
            pk[c / 2] = pack_p(p0, p1);
          }
        } else {
          const int vis = lim - kbase;
#pragma unroll
          for (int c = 0; c < BN; c += 2) {
            float a0, a1;
            f2_unpack(f2_fma(f2_pack(s[c], s[c + 1]), sl2x2, nbase2), a0, a1);
            const float p0 = c < vis ? ex2(a0) : 0.f, p1 = c + 1 < vis ? ex2(a1) : 0.f;
            acc2[(c >> 1) & (kAcc - 1)] = f2_add(acc2[(c >> 1) & (kAcc - 1)], f2_pack(p0, p1));
            pk[c / 2] = pack_p(p0, p1);
          }
        }
        for (int i = 0; i < 4; ++i) acc2[i] = f2_add(acc2[i], acc2[i + 4]);
        float acc[8];
        f2_unpack(acc2[0], acc[0], acc[1]);
        f2_unpack(acc2[1], acc[2], acc[3]);
        f2_unpack(acc2[2], acc[4], acc[5]);
        f2_unpack(acc2[3], acc[6], acc[7]);
        const float sum = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
        l = l * alpha + sum;
        if constexpr (kEarly) {
          // O_t += P_t(j-1) V has completed: O_t may be rescaled and P_t's buffer rewritten
          if (!first) {
            if (!warp_wait(bar(kBarPvDone + t), npv & 1, abort, p.status, p.wait_ns)) {
              ok = false;
              break;
            }
            ++npv;
            tc_fence_after();
          }
        }
        if (!first && __any_sync(0xffffffffu, alpha != 1.f)) {
          // O_t += P_t(j-1) V has completed (covered by the commit of S_t(j)).
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t u[32];
            tmem_ld32(o_col + 32 * c, u);
#pragma unroll
            for (int e = 0; e < 32; ++e) u[e] = __float_as_uint(__uint_as_float(u[e]) * alpha);
            tmem_st32(o_col + 32 * c, u);
          }
        }
        m = m_new;
        first = false;
        if constexpr (kFp8) {
          // P in E4M3 (p <= 2^8 < 448, the largest finite value), row r of the tile's
          // 128 x 128-byte buffer, 16-byte chunk c at chunk position c ^ (r mod 8) (the
          // 128-byte swizzle the descriptor declares). P_t's previous product has
          // completed (the wait above).
          uint8_t* prow = smem + Lay::kOffP + t * Lay::kPBytes + r * 128;
#pragma unroll
          for (int c16 = 0; c16 < 8; ++c16) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)  // pk[i]: the E4M3 pair of columns 2i, 2i + 1
              w[e] = pk[8 * c16 + 2 * e] | (pk[8 * c16 + 2 * e + 1] << 16);
            *reinterpret_cast<uint4*>(prow + ((c16 ^ (r & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
          }
          fence_proxy_async_smem();
        } else {
          tmem_st64(p_col, pk);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarPFull + t));
      }
      if (!ok) break;
      release_mask();
      // epilogue: O / l in bf16 and the row's logsumexp
      if (!warp_wait(bar(kEarly ? kBarPvDone + t : kBarOFull + t), (kEarly ? npv : no) & 1, abort, p.status, p.wait_ns)) {
        ok = false;
        break;
      }
      if (kEarly)
        ++npv;
      else
        ++no;
      tc_fence_after();
      const bool live = row < x.L;
      // a row the mask left with no key: O = 0, lse = -inf
      const float inv = (kMasked && l == 0.f) ? 0.f : (kFp8 ? p.v_descale : 1.f) / l;
      const int wrow0 = x.base + t * BM + q4 * 32;  // this warp's first row
      if (wrow0 + 32 <= x.L) {
        // all 32 rows of the warp lie in the sequence: stage each 64-column half in the
        // warp's slot (row `lane` at 128 lane, 16-byte chunk c at c ^ (lane mod 8): the
        // 128-byte swizzle of the O tensor map) and store it with one TMA box
        slot_store = true;
#pragma unroll
        for (int hh = 0; hh < D / 64; ++hh) {
          if (lane == 0) bulk_wait_read_all();  // the slot's previous store has read it
          __syncwarp();
#pragma unroll
          for (int c2 = 0; c2 < 2; ++c2) {
            uint32_t u[32];
            tmem_ld32(o_col + 64 * hh + 32 * c2, u);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              uint32_t w[4];
#pragma unroll
              for (int i = 0; i < 4; ++i)
                w[i] = pack_bf16x2(__uint_as_float(u[8 * e + 2 * i]) * inv, __uint_as_float(u[8 * e + 2 * i + 1]) * inv);
              const int chunk = 4 * c2 + e;
              *reinterpret_cast<uint4*>(slot + lane * 128 + ((chunk ^ (lane & 7)) << 4)) =
                  make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(&to, slot_s, 64 * hh, x.h, x.row0 + wrow0);
            bulk_commit_group();
          }
        }
      } else {
        __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.o) + ((size_t)(x.row0 + row) * p.Hq + x.h) * D;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t u[32];
          tmem_ld32(o_col + 32 * c, u);
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
      }
      if (live && p.lse) {
        const float lse = (kMasked && l == 0.f) ? -CUDART_INF_F : (m + log2f(l)) * kLn2;
        if (p.cu_seqlens)
          p.lse[(size_t)x.h * p.total_rows + x.row0 + row] = lse;
        else
          p.lse[((size_t)x.b * p.Hq + x.h) * p.N + row] = lse;
      }
    }
  }

  // the epilogue's TMA stores complete before the CTA (and its staging slots) goes away
  if (warp >= 4 && lane == 0) bulk_wait_all();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, int kMode>
cudaError_t launch_t(const PrefillParams& p, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                     const CUtensorMap& to, int num_sms, cudaStream_t stream) {
  using Lay = TcLayout<D, kMode>;
  auto kern = prefill_tc_kernel<D, kMode>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kBytes);
  if (e != cudaSuccess) return e;
  const long long pairs = (p.N + kRowsPerItem - 1) / kRowsPerItem;
  const long long items = (long long)p.B * p.Hq * pairs;
  if (items > 0x7fffffffLL) return cudaErrorInvalidValue;
  const int grid = (int)(items < num_sms ? items : num_sms);
  kern<<<grid, kThreads, Lay::kBytes, stream>>>(tq, tk, tv, to, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_tc(const PrefillParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                              const CUtensorMap& tv, const CUtensorMap& to, int num_sms, cudaStream_t stream) {
  if (p.block_mask) {
    if (p.d == 128) return launch_t<128, kModeSparse>(p, tq, tk, tv, to, num_sms, stream);
    return launch_t<64, kModeSparse>(p, tq, tk, tv, to, num_sms, stream);
  }
  if (p.block_table) {
    if (p.d == 128) return launch_t<128, kModePaged>(p, tq, tk, tv, to, num_sms, stream);
    return launch_t<64, kModePaged>(p, tq, tk, tv, to, num_sms, stream);
  }
  if (p.fp8) return p.d == 128 ? launch_t<128, kModeFp8>(p, tq, tk, tv, to, num_sms, stream) : cudaErrorInvalidValue;
  if (p.mask) {
    if (p.d == 128) return launch_t<128, kModeMasked>(p, tq, tk, tv, to, num_sms, stream);
    return launch_t<64, kModeMasked>(p, tq, tk, tv, to, num_sms, stream);
  }
  if (p.d == 128) return launch_t<128, kModeDense>(p, tq, tk, tv, to, num_sms, stream);
  return launch_t<64, kModeDense>(p, tq, tk, tv, to, num_sms, stream);
}

}  // namespace fattn
