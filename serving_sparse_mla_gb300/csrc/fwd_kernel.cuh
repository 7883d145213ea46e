// DSA sparse-MLA attention forward for sm_103a (cp.async gather + tcgen05).
//
// Computes, per query token t and head h over the token's top-k index list
// ("feat: add XTuner TileLang sparse MLA backend", Performance, Isolated
// sparse MLA forward: dqk=576, dv=512, topk=2048, BF16 Q/KV):
//
//   s_j   = sm_scale * q[t,h,:] . kv[r_j,:]              (576-wide latent rows)
//   LSE   = ln sum_j exp(s_j)                             (fp32, natural log)
//   out   = sum_j exp(s_j - LSE) * kv[r_j, 0:512]         (bf16)
//
// over the valid entries j (not -1 and inside the token's KV range; the
// TileLang page's Validation covers -1 padded lists).  A list with no valid
// entry gives out = 0 and LSE = -inf.  One latent KV head is shared by all
// query heads and its first 512 columns are the value ("[Feature] Add
// optional FlashMLA backend for DSA Sparse MLA", Runtime constraints:
// kv_group=1, value_dim=512).  The same kernel serves dense prefill, packed
// (cu_seqlens) prefill and the paged BF16 cache (TileLang page, Summary);
// only the index -> row mapping differs.
//
// Work decomposition: a persistent grid of at most one CTA per SM (each
// takes ~225 KB of shared memory).  A unit of work is one token's list for
// one group of up to 64 heads; prefill deals whole units round-robin to the
// CTAs, decode cuts the units' lists, laid end to end, into one equal range
// per CTA; the CTA that writes a cut unit's last piece merges its pieces.
// Every role of a CTA walks the same sequence of items, so the producers
// gather the next item while the consumers finish the current one.  The
// index list is walked in blocks of 64 entries (64 gathered rows = 72 KB, so
// two to three blocks fit in shared memory and the gather of the next blocks
// overlaps the math of the current one); a block with no valid entry is
// skipped.  Per block:
//
//   warps 0..3         map the block's indices to KV rows (every warp maps
//   (producers)        all 64 entries, so all agree on the block-skip and the
//                      validity mask without a barrier) and copy the rows
//                      into shared memory with 16-byte cp.async, 128B-swizzled:
//                      four 64x128 "pair" tiles for columns 0..511 (the value
//                      part) and one 64x64 tile for the rope columns; each
//                      warp copies its 16 rows of every tile.  Masked rows are
//                      zero-filled (source size 0) and never read.  Producers
//                      never wait on their own copies: the hardware arrives on
//                      the tile's full barrier when a thread's copies have
//                      landed, and the MMA thread, after acquiring the tile,
//                      issues fence.proxy.async before the tensor core reads
//                      it.  On GB300 this gathers random 1152-B rows ~6x
//                      faster than TMA tile::gather4 (13.9 vs 2.2 TB/s from
//                      L2, 5.3 vs 2.2 TB/s from HBM).
//   warps 4, 9 and    three threads issue tcgen05.mma (kind::f16, fp32 in
//   the last warp      TMEM): two split QK^T (value pairs 0,1 + rope / pairs
//   (MMA)              2,3, into two partial S^T) and one issues P.V as soon as
//                      P^T is ready; one issuer sustains ~59 cycles per MMA on
//                      GB300, several more in aggregate:
//                        S^T[64 x N]   = K_blk[64 x 576] . Q^T[576 x N]   (M=64)
//                        O^T[512 x N] += V^T[512 x 64]  . P^T[64 x N]    (M=128)
//                      (swap-AB: kv rows are M and heads are N, so 8 heads
//                      cost N=16 instead of a 64-row pad).  V^T is the same
//                      gathered tile read through an MN-major descriptor.  S
//                      is double-buffered, so QK of the next block runs while
//                      the softmax works on the current one.
//   warps 5..8         the M=64 result sits in lanes 32*(i/16) + i%16, so
//   (+ 10..13 for      lanes 0..15 of each warp own one kv row each; a group
//   64 heads;          of 4 warps owns up to 32 heads (two groups for 64 heads,
//   softmax)           each with its own named barrier).  Per row: add the
//                      two partial S^T rows, mask, reduce the per-head block
//                      max across the 64 rows (warp transpose-reduce plus a
//                      shared-memory step), keep a lazily updated running max
//                      (O is rescaled only when a head's max grows by more
//                      than 2^8, after the previous P.V has completed), write
//                      P^T = exp2(s - m) as bf16 into the block's rope slot,
//                      and at the end normalise O^T and write out / LSE.
//
// All waits are bounded (see ptx.cuh); a timed-out CTA records an error in
// the device error word, drains its in-flight copies and MMAs, frees TMEM
// and returns.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "ptx.cuh"

namespace smla {

constexpr int kDqk = 576;
constexpr int kDv = 512;
constexpr int kBlk = 64;                     // index entries (kv rows) per block
constexpr int kChunkBytes = kBlk * 128;      // 64 rows x 64 bf16 columns
constexpr int kPairBytes = 2 * kChunkBytes;  // 64 rows x 128 columns
constexpr int kInfoDepth = 8;
constexpr int kProducerWarps = 4;
constexpr int kMmaWarp = 4;                  // QK^T issuer, part 0 (also owns the TMEM allocation)
constexpr int kMmaWarpB = 9;                 // QK^T issuer, part 1
// P.V issuer: the warp after the softmax groups (10 or 14).
// Softmax group g (4 warps, one per TMEM lane quarter) owns heads
// [32 g, 32 g + 32): warps 5..8 for g = 0, warps 10..13 for g = 1.
__host__ __device__ constexpr int softmax_warp0(int g) { return g == 0 ? 5 : 10; }
constexpr float kLazyRescale = 8.0f;         // log2 units
constexpr int kMaxSmem = 232448;

// kCausal: dense rows without an index tensor; entry e of token t's list is
// position e while e <= t + causal_off (every causal position selected, the
// short-prefill case of "feat: add XTuner TileLang sparse MLA backend",
// Summary), else masked.
// kPagedFp8: the paged layout over an FP8 cache (656-byte slots: 512 e4m3
// codes, four fp32 tile scales, 64 bf16 rope values).  At 16 heads the
// tensor cores contract the codes and the tile scales are applied to the
// partial scores and to P (Layout kRaw); at 32 and 64 heads the rows are
// dequantized to bf16 as they are gathered.
enum Mode : int { kDense = 0, kVarlen = 1, kPaged = 2, kCausal = 3, kPagedFp8 = 4 };

// FP8 cache slot layout (the FP8 sparse-decode cache published with
// DeepSeek-V3.2's FlashMLA kernels; the pages name the path, not its format).
constexpr int kFp8SlotBytes = 656;
constexpr int kFp8ScaleOff = 512;
constexpr int kFp8RopeOff = 528;

// How units (token x head group) are dealt to the persistent CTAs:
//   kWholeUnits   CTA c runs units c, c + G, c + 2G, ... whole (prefill).
//   kBlockRanges  the units' index lists, laid end to end as T = units x nb
//                 blocks of 64 entries, are cut into G equal ranges, one per
//                 CTA (decode: a few long lists spread over every SM).  A unit
//                 cut between CTAs leaves a partial result per piece; the CTA
//                 that writes a unit's last piece merges them (merge_row).
enum Sched : int { kWholeUnits = 0, kBlockRanges = 1 };

enum ErrCode : int { kErrProducerWait = 0x101, kErrMmaWait = 0x201, kErrSoftmaxWait = 0x301 };

struct FwdParams {
  const __nv_bfloat16* q;   // [n_tok, h_q, 576]
  const __nv_bfloat16* kv;  // [n_rows, 576] (paged: [num_blocks * page_size, 576])
  const int32_t* indices;   // [n_tok, topk]
  __nv_bfloat16* out;       // [n_tok, h_q, 512]
  float* lse;               // [n_tok, h_q]
  float* part_o;            // [2 * ctas, part_rows, 512]  (kBlockRanges)
  float* part_lse;          // [2 * ctas, part_rows]
  const int32_t* cu_q;      // varlen: [batch+1]
  const int32_t* cu_kv;     // varlen: [batch+1]
  const int32_t* block_table;  // paged: [batch, max_blocks]
  const int32_t* seqlens;      // paged: [batch]
  int n_tok, h_q, topk, mode;
  int n_rows;               // rows of kv
  int s_kv, batch, s_next, page_size, max_blocks, num_blocks;
  int causal_off;           // kCausal: s_kv - s_q (query t sits at position t + causal_off)
  int sched;                // kWholeUnits or kBlockRanges
  int groups;               // head groups of up to 64 (a unit is one token x one group)
  int nb;                   // 64-entry blocks per index list
  int ctas;                 // CTAs of the (persistent) grid
  int part_rows;            // head rows per partial slot: min(h_q, 64)
  float scale_log2;         // sm_scale * log2(e)
  float sm_scale;
  // backward only: out and lse above are the forward's results (inputs)
  const __nv_bfloat16* dout;  // [n_tok, h_q, 512]
  float* dq;                  // [n_tok, h_q, 576]
  float* dkv;                 // [n_rows, 576], accumulated
  int32_t* valid_count;       // debug count export: [n_tok], zeroed, accumulated
  int32_t* merge_count;       // kBlockRanges: pieces written per (unit, softmax group), zeroed before the launch
  unsigned long long timeout_ns;
};

__device__ int g_device_error;

// kBlockRanges: CTA c covers flattened blocks [range_start(c), range_start(c+1)).
__host__ __device__ inline long long range_start(int c, long long total, int ctas) {
  return static_cast<long long>(c) * total / ctas;
}
// The CTA whose range holds flattened block x (0 <= x < total).
__host__ __device__ inline int range_cta(long long x, long long total, int ctas) {
  return static_cast<int>(((x + 1) * ctas - 1) / total);
}

// One piece of work: blocks [jb, je) of a unit's index list.  slot < 0: the
// CTA runs the whole unit and writes out / LSE; else it writes a partial
// result to slot 2c (its first item) or 2c + 1 (its last item).
struct Item {
  int unit, jb, je, slot;
};

struct ItemIter {
  long long x;   // kBlockRanges: next flattened block of this CTA
  int k;         // items handed out so far
};

__device__ __forceinline__ ItemIter items_begin(const FwdParams& p) {
  ItemIter it;
  it.k = 0;
  it.x = p.sched == kBlockRanges
             ? range_start(static_cast<int>(blockIdx.x), static_cast<long long>(p.n_tok) * p.groups * p.nb, p.ctas)
             : 0;
  return it;
}

// Every role of a CTA walks the same item sequence with its own iterator.
__device__ __forceinline__ bool next_item(const FwdParams& p, ItemIter& it, Item& out) {
  const int c = static_cast<int>(blockIdx.x);
  const long long units = static_cast<long long>(p.n_tok) * p.groups;
  if (p.sched == kWholeUnits) {
    const long long u = c + static_cast<long long>(it.k) * p.ctas;
    if (u >= units) return false;
    out.unit = static_cast<int>(u);
    out.jb = 0;
    out.je = p.nb;
    out.slot = -1;
    ++it.k;
    return true;
  }
  const long long total = units * p.nb;
  const long long end = range_start(c + 1, total, p.ctas);
  if (it.x >= end) return false;
  const long long u = it.x / p.nb;
  const long long ub = u * p.nb;
  out.unit = static_cast<int>(u);
  out.jb = static_cast<int>(it.x - ub);
  out.je = static_cast<int>(min(static_cast<long long>(p.nb), end - ub));
  const bool whole = range_cta(ub, total, p.ctas) == range_cta(ub + p.nb - 1, total, p.ctas);
  out.slot = whole ? -1 : 2 * c + (it.k == 0 ? 0 : 1);
  it.x = ub + out.je;
  ++it.k;
  return true;
}

// kRaw: the FP8 cache at 16 heads.  The producers copy each value tile's
// raw e4m3 codes (64 rows x 128 codes) into the second 64-column chunk of its
// value slot, and converter warps rewrite the slot in place as bf16 values
// code * 2^-120 (exact, no scale applied), each warp its own rows, so the
// conversion can be spread over more warps than the producers' row groups.
// The tensor core then contracts the codes:
// QK^T keeps one partial S^T per 128-column scale tile (and one for the
// rope), which the softmax combines with the rows' tile scales, and P.V
// takes, per value tile t, P^T scaled by the rows' scale of tile t and 2^88
// (four bf16 tiles that fill the block's rope slot; O^T then holds the
// output times 2^-32).  The rows' scales (1 KB per
// block) ride with the rope tile into a scale ring indexed like the rope
// ring, so the rope slot's release also releases them.
template <int N, bool kRaw = false>
struct Layout {
  static_assert(N == 16 || N == 32 || N == 64, "head group width");
  static_assert(!kRaw || N == 16, "codes contracted unscaled: 16 heads only");
  static constexpr bool kRawCodes = kRaw;
  static constexpr int kNV = N == 64 ? 8 : (N == 32 ? 10 : 11);  // value pair-tile ring
  static constexpr int kNR = N == 64 ? 2 : 3;                     // rope / P^T ring
  static constexpr int kNSc = kRaw ? kNR : 0;                     // per-block scale ring (slot = rope slot)
  static constexpr int kPRow = N * 2;                             // bytes of one P^T row
  static constexpr uint32_t kPSwz = N == 64 ? SWZ_128B : (N == 32 ? SWZ_64B : SWZ_32B);
  // TMEM: the partial S^T (2 parts, or kRaw 5 tiles, double-buffered), then O^T
  static constexpr int kSParts = kRaw ? 5 : 2;
  static constexpr int kOCol = 2 * kSParts * N;
  static constexpr int kTmemCols = kRaw ? 256 : (N == 64 ? 512 : (N == 32 ? 256 : 128));
  static_assert(kOCol + 4 * N <= kTmemCols, "TMEM columns");
  static constexpr int kGroups = N == 64 ? 2 : 1;                 // softmax groups
  static constexpr int kHG = N / kGroups;                         // heads per group (<= 32)
  static constexpr int kPvWarp = 6 + 4 * kGroups;
  static constexpr int kThreads = (kPvWarp + 1) * 32;
  static constexpr int kQOff = 0;
  static constexpr int kVOff = 9 * N * 128;
  static constexpr int kROff = kVOff + kNV * kPairBytes;
  static constexpr int kScOff = kROff + kNR * kChunkBytes;
  static constexpr int kMiscOff = kScOff + kNSc * 1024;
  static_assert(kBlk * kPRow * (kRaw ? 4 : 1) <= kChunkBytes, "P^T (kRaw: its four scaled tiles) fits in a rope slot");
  // Block n+2's last value tile reuses a slot that P.V of block n frees, so
  // the softmax of block n+2 cannot finish before P.V(n) has started; that
  // keeps every double-buffered phase wait (p_full, s_full) within one phase.
  static_assert(kNV >= 8 && kNV <= 11, "value ring must span 2 to 2.75 blocks");
  static_assert(kNR >= 2, "P^T of the next block needs its own rope slot");
};

// FP8 cache at 16 heads per CTA: eight converter warps after the P.V warp,
// two per value tile, widen each tile's codes in place in its value slot as
// they land (the other widths dequantize in the producer warps, one block
// behind their copies, in place in the value slots).
template <int N, bool kFp8>
__host__ __device__ constexpr int conv_warps() { return (kFp8 && N == 16) ? 8 : 0; }
template <int N, bool kFp8>
__host__ __device__ constexpr int fwd_threads() { return Layout<N>::kThreads + 32 * conv_warps<N, kFp8>(); }
// The shared-memory layout of the kernel instantiation <N, kFp8>.
template <int N, bool kFp8>
using LayoutFor = Layout<N, kFp8 && N == 16>;

struct __align__(16) Misc {
  uint64_t v_full[12], v_empty[12];
  uint64_t raw_full[12];   // FP8 with converter warps: a value slot's raw codes have landed
  uint64_t rp_full[3], rp_empty[3];
  uint64_t info_full[kInfoDepth], info_empty[kInfoDepth];
  uint64_t q_full, q_empty, s_full[2][2], p_full[2], o_full, drain[3], cand_full;
  int32_t info_blk[kInfoDepth];
  uint32_t info_mask[kInfoDepth][2];
  uint32_t cand[2][kProducerWarps];
  float red[4][64];
  float rsum[4][64];
  float mrun[64];
  float alpha[64];
  float fin[64];
  uint32_t tmem_base;
  int abort_flag;
  int prior_error;
  int merge_pieces[2];       // per softmax group: pieces of the unit to merge here (0: none)
  int merge_slot[2][32];     // their partial slots
};

template <int N, bool kFp8 = false>
constexpr int smem_bytes() {
  return LayoutFor<N, kFp8>::kMiscOff + static_cast<int>(sizeof(Misc)) + 1024;
}
static_assert(smem_bytes<64>() <= kMaxSmem, "smem budget (64 heads)");
static_assert(smem_bytes<32>() <= kMaxSmem, "smem budget (32 heads)");
static_assert(smem_bytes<16>() <= kMaxSmem, "smem budget (16 heads)");
static_assert(smem_bytes<16, true>() <= kMaxSmem, "smem budget (16 heads, FP8 cache)");

// ------------------------------------------------------------------ helpers

struct TokCtx {
  int kv_lo;
  int kv_len;
  const int32_t* table;
};

__device__ __forceinline__ TokCtx token_context(const FwdParams& p, int tok) {
  TokCtx c;
  c.table = nullptr;
  if (p.mode == kDense || p.mode == kCausal) {
    c.kv_lo = 0;
    c.kv_len = p.s_kv;
  } else if (p.mode == kVarlen) {
    int lo = 0, hi = p.batch;  // largest b with cu_q[b] <= tok
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(p.cu_q + mid) <= tok) lo = mid; else hi = mid;
    }
    c.kv_lo = __ldg(p.cu_kv + lo);
    c.kv_len = __ldg(p.cu_kv + lo + 1) - c.kv_lo;
  } else {   // kPaged, kPagedFp8
    const int b = tok / p.s_next;
    c.kv_lo = 0;
    c.kv_len = __ldg(p.seqlens + b);
    c.table = p.block_table + static_cast<size_t>(b) * p.max_blocks;
  }
  return c;
}

// Entry e (< topk) of a token's index list: read from the list, or in the
// causal mode the position itself while it is at or before the token's own
// position `last` (no memory read).
template <bool kCausalList>
__device__ __forceinline__ int index_at(const int32_t* irow, int last, int e) {
  if constexpr (kCausalList) return e <= last ? e : -1;
  else return __ldg(irow + e);
}

// The paged layouts' block-table entry of an index entry's page (-1 when the
// entry is outside the token's range or its page past the table's width);
// 0 for the other layouts.  Split from map_entry so that the producer can
// load the next block's entries while it issues the current block's copies.
__device__ __forceinline__ int table_entry(const FwdParams& p, const TokCtx& c, int idx) {
  if (!(p.mode == kPaged || p.mode == kPagedFp8)) return 0;
  if (idx < 0 || idx >= c.kv_len) return -1;
  const int pg = idx / p.page_size;
  if (pg >= p.max_blocks) return -1;
  return __ldg(c.table + pg);
}

// KV row read by one index entry (blk: its table_entry), or -1 when the
// entry is masked.
__device__ __forceinline__ int map_entry(const FwdParams& p, const TokCtx& c, int idx, int blk) {
  if (idx < 0 || idx >= c.kv_len) return -1;
  int row;
  if (p.mode == kPaged || p.mode == kPagedFp8) {
    if (blk < 0 || blk >= p.num_blocks) return -1;
    row = blk * p.page_size + idx % p.page_size;
  } else {
    row = c.kv_lo + idx;
  }
  return (row >= 0 && row < p.n_rows) ? row : -1;
}

__device__ __forceinline__ void raise_error(Misc& m, int code) {
  *reinterpret_cast<volatile int*>(&m.abort_flag) = 1;
  atomicCAS(&g_device_error, 0, code);
}

// Transposing butterfly over the warp: lane l ends with the reduction (over
// the 32 lanes) of a contiguous run of heads and writes it to dst[head].
template <int N, bool kMax>
__device__ __forceinline__ void warp_xreduce(float (&v)[N], int lane, float* dst) {
  int cnt = N;
  int base = 0;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    if (cnt > 1) {
      const int half = cnt >> 1;
      const bool upper = (lane & off) != 0;
#pragma unroll
      for (int i = 0; i < N / 2; ++i) {
        if (i < half) {
          const float send = upper ? v[i] : v[i + half];
          const float keep = upper ? v[i + half] : v[i];
          const float recv = __shfl_xor_sync(0xffffffffu, send, off);
          v[i] = kMax ? fmaxf(keep, recv) : keep + recv;
        }
      }
      if (upper) base += half;
      cnt = half;
    } else {
      const float recv = __shfl_xor_sync(0xffffffffu, v[0], off);
      v[0] = kMax ? fmaxf(v[0], recv) : v[0] + recv;
    }
  }
#pragma unroll
  for (int i = 0; i < N; ++i)
    if (i < cnt) dst[base + i] = v[i];
}

// The same butterfly within each 16-lane half of the warp (the halves hold
// different heads of the same rows); dst is the half's first head.  kOff0 < 8
// continues a butterfly whose first levels were taken already (v then holds
// the heads from dst on).
template <int V, bool kMax, int kOff0 = 8>
__device__ __forceinline__ void half_xreduce(float (&v)[V], int lane, float* dst) {
  int cnt = V;
  int base = 0;
#pragma unroll
  for (int off = kOff0; off >= 1; off >>= 1) {
    if (cnt > 1) {
      const int half = cnt >> 1;
      const bool upper = (lane & off) != 0;
#pragma unroll
      for (int i = 0; i < V / 2; ++i) {
        if (i < half) {
          const float send = upper ? v[i] : v[i + half];
          const float keep = upper ? v[i + half] : v[i];
          const float recv = __shfl_xor_sync(0xffffffffu, send, off);
          v[i] = kMax ? fmaxf(keep, recv) : keep + recv;
        }
      }
      if (upper) base += half;
      cnt = half;
    } else {
      const float recv = __shfl_xor_sync(0xffffffffu, v[0], off);
      v[0] = kMax ? fmaxf(v[0], recv) : v[0] + recv;
    }
  }
#pragma unroll
  for (int i = 0; i < V; ++i)
    if (i < cnt) dst[base + i] = v[i];
}

// bar.sync over the 128 threads of one softmax group (named barrier `id`),
// returning the OR of `pred`.
__device__ __forceinline__ bool bar_red_or_128(uint32_t id, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(id)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

__device__ __forceinline__ void cp_async_arrive_on(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Codes 2k and 2k + 1 of four e4m3 codes w (code i in byte i) as bf16x2
// holding code * 2^-120 exactly: a bf16 whose exponent field is the e4m3's
// exponent field and whose top three mantissa bits are the e4m3's mantissa
// reads the e4m3 exponent bias 7 against 127, for subnormals (exponent field
// 0) as well.  The byte permute places each code in the low byte of its
// 16-bit lane with its sign replicated in the high byte; shifted left by four
// bits, the lane holds the sign at bit 15 and exponent and mantissa at bits
// 10..4, and the mask clears the rest (including what the shift carries from
// the low lane into the high lane's bits 0..3).
template <int K>
__device__ __forceinline__ uint32_t e4m3x2_bf16x2_shifted(uint32_t w) {
  uint32_t x;
  asm("prmt.b32 %0, %1, 0, %2;" : "=r"(x) : "r"(w), "n"(K == 0 ? 0x9180 : 0xB3A2));
  return (x << 4) & 0x87F087F0u;
}

// Two e4m3 codes (the low byte first) times a scale -> bf16x2 (round to
// nearest even): e4m3 -> f16 is exact, the product is formed in fp32.
__device__ __forceinline__ uint32_t e4m3x2_scaled_bf16x2(uint32_t two_codes, float scale) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<unsigned short>(two_codes)));
  const __half2 h = *reinterpret_cast<const __half2*>(&h2);
  const float2 f = __half22float2(h);
  return pack_bf16x2(f.x * scale, f.y * scale);
}

// ------------------------------------------------------------------ producer

// FP8 gather, second half: block nb's four value tiles, whose raw e4m3 codes
// (in each slot's second chunk) and tile scales (in the first tile's first
// chunk, two rows per row group of 16) have landed (wait_tile(u, slot)
// returns once tile u's have, false on a timeout), are dequantized in place
// into the 128B-swizzled bf16 layout the MMA descriptors read; then each
// tile's full barrier gets this thread's arrival.  Row group `warp` (rows
// 16 warp .. 16 warp + 15): a lane converts 16 codes of one row per value
// tile, the bytes that the producer lane of the same position copied.  The
// scales are read before any store (the first tile's stores overwrite them),
// and every row group's codes are read before its stores (a row's bf16
// second chunk overwrites its codes).
template <class L, class M, class Wait>
__device__ __forceinline__ bool fp8_convert_block(M& m, uint32_t vbase, int nb, int warp, int sel, int piece,
                                                  Wait&& wait_tile) {
  const int ch = piece >> 2, pc = (piece & 3) * 2;
  const uint8_t* gbase = reinterpret_cast<const uint8_t*>(&m) - smem_u32(&m);   // generic address of shared offset 0
  float sc[4][4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const uint32_t s = (static_cast<uint32_t>(nb) * 4u + static_cast<uint32_t>(u)) % L::kNV;
    if (!wait_tile(u, s)) return false;
    const uint32_t dst = vbase + s * kPairBytes;
    const uint8_t* tile = gbase + dst;
    if (u == 0) {
#pragma unroll
      for (int it = 0; it < 4; ++it) {
        const float4 f = *reinterpret_cast<const float4*>(tile + warp * 2048 + (it * 4 + sel) * 16);
        sc[it][0] = f.x;
        sc[it][1] = f.y;
        sc[it][2] = f.z;
        sc[it][3] = f.w;
      }
    }
    // The row group's codes of this tile (all four row sets in flight), then
    // the stores: the second chunk's bf16 rows overwrite the codes, and the
    // first tile's first chunk the scales.
    uint4 c[4];
#pragma unroll
    for (int it = 0; it < 4; ++it)
      c[it] = *reinterpret_cast<const uint4*>(tile + kChunkBytes + (warp * 16 + it * 4 + sel) * 128 + piece * 16);
    __syncwarp();
#pragma unroll
    for (int it = 0; it < 4; ++it) {
      const int r = warp * 16 + it * 4 + sel;
      const float f = sc[it][u];
      // 16 codes: columns 128 u + 16 piece .. + 15 = chunk piece / 4, 8-column
      // pieces 2 (piece % 4) and 2 (piece % 4) + 1 of row r
      const uint32_t at = dst + ch * kChunkBytes + r * 128;
      st_shared_v4(at + ((pc ^ (r & 7)) << 4), e4m3x2_scaled_bf16x2(c[it].x, f),
                   e4m3x2_scaled_bf16x2(c[it].x >> 16, f), e4m3x2_scaled_bf16x2(c[it].y, f),
                   e4m3x2_scaled_bf16x2(c[it].y >> 16, f));
      st_shared_v4(at + (((pc + 1) ^ (r & 7)) << 4), e4m3x2_scaled_bf16x2(c[it].z, f),
                   e4m3x2_scaled_bf16x2(c[it].z >> 16, f), e4m3x2_scaled_bf16x2(c[it].w, f),
                   e4m3x2_scaled_bf16x2(c[it].w >> 16, f));
    }
    // the tile's bf16 rows are written: order them before the tensor core's
    // reads (async proxy) and arrive on its full barrier
    fence_proxy_async_smem();
    mbar_arrive(smem_u32(&m.v_full[s]));
  }
  return true;
}

// The gather producer, shared with the backward kernel: L gives the shared
// memory layout (ring sizes and offsets), M the barrier block (same member
// names), and kRows also publishes each block's 64 KV rows (entry r of the
// block in info_rows[k][r], -1 when masked) for consumers that scatter by row.
// kCount walks the same windows, block skips, row mapping and validity
// ballots but copies and publishes nothing: it adds each item's number of
// valid entries to p.valid_count[token] (the debug count export).
// kFp8 gathers FP8 cache slots (kPagedFp8) and dequantizes them to bf16.
// kConv (with kFp8): converter warps dequantize the tiles; the producer only
// copies, and each value tile's raw codes arrive on raw_full.
template <int N, class L, class M, bool kRows, bool kCausalList = false, bool kCount = false, bool kFp8 = false,
          bool kConv = false>
__device__ bool run_producer_t(const FwdParams& p, M& m, uint8_t* sbase) {
  const int warp = static_cast<int>(threadIdx.x >> 5);   // 0..3
  const int lane = static_cast<int>(lane_id());
  const volatile int* ab = &m.abort_flag;
  const uint32_t vbase = smem_u32(sbase + L::kVOff);
  const uint32_t rbase = smem_u32(sbase + L::kROff);
  const int piece = lane & 7;
  const int sel = lane >> 3;
  // Every warp maps the whole block (entries 2*lane, 2*lane+1) so all agree
  // on the skip decision and on ring positions without a barrier; each warp
  // then copies its own 16 rows of every tile.
  int n = 0;     // blocks issued: position in the tile rings
  int ni = 0;    // info entries published: blocks and per-item end markers
  int win = 0;   // index windows scanned (phase of cand_full)
  int counted = 0;   // kCount: valid entries of the current item
  ItemIter iter = items_begin(p);
  Item item;
  uint64_t deadline = 0;
  while (next_item(p, iter, item)) {
    deadline = global_timer_ns() + p.timeout_ns;   // every wait of this item is bounded from here
    const int tok = item.unit / p.groups;
    const int jb = item.jb, je = item.je;
    const TokCtx ctx = token_context(p, tok);
    const int32_t* irow = kCausalList ? nullptr : p.indices + static_cast<size_t>(tok) * p.topk;
    const int last = tok + p.causal_off;   // kCausal only
    for (int wb = jb; wb < je; wb += 32, ++win) {
      // Candidate blocks of this window of up to 32: a block none of whose
      // entries lies in [0, kv_len) is skipped without mapping its rows (a
      // causal list is mostly -1 padding for early tokens).  Each warp scans 8
      // blocks with 16 coalesced loads in flight per lane; the four masks meet
      // in shared memory.  The loads also bring the list into L1 for the row
      // mapping below.
      const int we = min(je, wb + 32);
      uint32_t cand;
      {
        const int b0 = wb + warp * 8;
        int v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int blk = b0 + (i >> 1);
          const int e = blk * kBlk + (i & 1) * 32 + lane;
          v[i] = (blk < we && e < p.topk) ? index_at<kCausalList>(irow, last, e) : -1;
        }
        uint32_t bits = 0;
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
          const bool c = (v[i] >= 0 && v[i] < ctx.kv_len) || (v[i + 1] >= 0 && v[i + 1] < ctx.kv_len);
          if (__ballot_sync(0xffffffffu, c) != 0u) bits |= 1u << (i >> 1);
        }
        if (lane == 0) {
          m.cand[win & 1][warp] = bits << (warp * 8);
          mbar_arrive(smem_u32(&m.cand_full));
        }
        const bool ok = mbar_wait(smem_u32(&m.cand_full), static_cast<uint32_t>(win) & 1u, deadline, ab);
        if (!__all_sync(0xffffffffu, ok)) return false;
        cand = 0;
#pragma unroll
        for (int w = 0; w < kProducerWarps; ++w) cand |= *reinterpret_cast<volatile uint32_t*>(&m.cand[win & 1][w]);
      }
      int j_next = cand != 0u ? wb + __ffs(static_cast<int>(cand)) - 1 : -1;
      int idx_next[2], tbl_next[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int e = j_next * kBlk + lane * 2 + i;
        idx_next[i] = (j_next >= 0 && e < p.topk) ? index_at<kCausalList>(irow, last, e) : -1;
        tbl_next[i] = table_entry(p, ctx, idx_next[i]);
      }
      while (j_next >= 0) {
        const int j = j_next;
        cand &= cand - 1u;
        j_next = cand != 0u ? wb + __ffs(static_cast<int>(cand)) - 1 : -1;
        int rows[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) rows[i] = map_entry(p, ctx, idx_next[i], tbl_next[i]);
        // The next candidate's indices, and (paged) its table entries: their
        // loads are in flight while this block's copies are issued.
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int e = j_next * kBlk + lane * 2 + i;
          idx_next[i] = (j_next >= 0 && e < p.topk) ? index_at<kCausalList>(irow, last, e) : -1;
          tbl_next[i] = table_entry(p, ctx, idx_next[i]);
        }
        const uint32_t bal0 = __ballot_sync(0xffffffffu, rows[0] >= 0);
        const uint32_t bal1 = __ballot_sync(0xffffffffu, rows[1] >= 0);
        if ((bal0 | bal1) == 0u) continue;
        if constexpr (kCount) {
          counted += __popc(bal0) + __popc(bal1);
          continue;
        }

        if (warp == 0) {
          const int k = ni % kInfoDepth;
          const bool ok = mbar_wait(smem_u32(&m.info_empty[k]), ((ni / kInfoDepth) & 1) ^ 1, deadline, ab);
          if (!__all_sync(0xffffffffu, ok)) return false;
          if constexpr (kRows) {
            m.info_rows[k][2 * lane] = rows[0];
            m.info_rows[k][2 * lane + 1] = rows[1];
            __syncwarp();
          }
          if (lane == 0) {
            m.info_blk[k] = j;
            m.info_mask[k][0] = bal0;
            m.info_mask[k][1] = bal1;
            mbar_arrive(smem_u32(&m.info_full[k]));
          }
        }
        // This warp copies block rows 16*warp + 4*it + sel; entry r of the block
        // sits in lane r / 2 as rows[r % 2].
        int myrow[4];
#pragma unroll
        for (int it = 0; it < 4; ++it) {
          const int r = warp * 16 + it * 4 + sel;
          const int r0 = __shfl_sync(0xffffffffu, rows[0], r >> 1);
          const int r1 = __shfl_sync(0xffffffffu, rows[1], r >> 1);
          myrow[it] = (r & 1) ? r1 : r0;
        }
        // Tile order: value pairs 0 and 1, the rope tile, pairs 2 and 3 -- the
        // QK^T part that needs pairs 0,1 and the rope can start after 3 tiles.
        auto tile = [&](int step, uint32_t& empty, uint32_t& full, uint32_t& par, uint32_t& dst, int& first_chunk,
                        int& n_chunks) {
          const int u = step < 2 ? step : (step == 2 ? 4 : step - 1);
          if (u < 4) {
            // (FP8 with converter warps: the raw codes' arrival goes to
            // raw_full, the converters arrive on v_full)
            const uint32_t vi = static_cast<uint32_t>(n) * 4u + static_cast<uint32_t>(u);
            const uint32_t s = vi % L::kNV;
            empty = smem_u32(&m.v_empty[s]);
            if constexpr (kConv) full = smem_u32(&m.raw_full[s]);
            else full = smem_u32(&m.v_full[s]);
            par = (vi / L::kNV) & 1u;
            dst = vbase + s * kPairBytes;
            first_chunk = 2 * u;
            n_chunks = 2;
          } else {
            const uint32_t rs = static_cast<uint32_t>(n) % L::kNR;
            empty = smem_u32(&m.rp_empty[rs]);
            full = smem_u32(&m.rp_full[rs]);
            par = (static_cast<uint32_t>(n) / L::kNR) & 1u;
            dst = rbase + rs * kChunkBytes;
            first_chunk = 8;
            n_chunks = 1;
          }
        };
        // One tile's copies into its (free) slot, then the arrival on its full
        // barrier: cp.async with a hardware arrival, or (FP8 value tiles)
        // dequantize, store, fence for the tensor core's proxy and arrive.
        auto copy_tile = [&](int step, uint32_t full, uint32_t dst, int first_chunk, int n_chunks) {
          const int u = step < 2 ? step : (step == 2 ? 4 : step - 1);
          if constexpr (kFp8) {
            if (u < 4) {
              // Raw e4m3 codes of the tile's 128 columns (row r at r * 128,
              // unswizzled) into the value slot's second 64-column chunk.
              // kConv: converted in place by the converter warps once raw_full
              // completes (the rows' scales go with the rope tile).  Else with
              // the first value tile the rows' four tile scales (16 bytes a
              // row) in the first two rows of this row group in its first
              // chunk, converted in place by this warp one block later
              // (fp8_convert_block).  Masked rows are zero-filled (codes and
              // scales 0: a zero row).
              const uint32_t code_dst = dst + kChunkBytes;
              const uint32_t sc_dst = dst + static_cast<uint32_t>(warp) * 2048u;
#pragma unroll
              for (int it = 0; it < 4; ++it) {
                const int r = warp * 16 + it * 4 + sel;
                const int src_row = myrow[it];
                const uint8_t* slot_src = reinterpret_cast<const uint8_t*>(p.kv) +
                                          static_cast<size_t>(src_row < 0 ? 0 : src_row) * kFp8SlotBytes;
                cp_async_16(code_dst + r * 128 + piece * 16, slot_src + u * 128 + piece * 16, src_row < 0 ? 0u : 16u);
                if (!kConv && u == 0 && piece == 0)
                  cp_async_16(sc_dst + (it * 4 + sel) * 16, slot_src + kFp8ScaleOff, src_row < 0 ? 0u : 16u);
              }
              if constexpr (kConv) cp_async_arrive_on(full);
              return;
            }
          }
          for (int c = 0; c < n_chunks; ++c) {
#pragma unroll
            for (int it = 0; it < 4; ++it) {
              const int r = warp * 16 + it * 4 + sel;
              const int src_row = myrow[it];
              const void* src;
              if constexpr (kFp8)   // the rope tile: 64 bf16 values after the codes and scales
                src = reinterpret_cast<const uint8_t*>(p.kv) +
                      static_cast<size_t>(src_row < 0 ? 0 : src_row) * kFp8SlotBytes + kFp8RopeOff + piece * 16;
              else
                src = p.kv + static_cast<size_t>(src_row < 0 ? 0 : src_row) * kDqk + (first_chunk + c) * 64 + piece * 8;
              cp_async_16(dst + c * kChunkBytes + r * 128 + ((piece ^ (r & 7)) << 4), src, src_row < 0 ? 0u : 16u);
            }
          }
          if constexpr (kConv) {
            // with the rope tile, the rows' four tile scales (16 bytes a row,
            // row r at r * 16) into the scale slot of the block's rope slot
            if (piece == 0) {
              const uint32_t sc_dst = smem_u32(sbase + L::kScOff) + (static_cast<uint32_t>(n) % L::kNR) * 1024u;
#pragma unroll
              for (int it = 0; it < 4; ++it) {
                const int r = warp * 16 + it * 4 + sel;
                const int src_row = myrow[it];
                cp_async_16(sc_dst + r * 16,
                            reinterpret_cast<const uint8_t*>(p.kv) +
                                static_cast<size_t>(src_row < 0 ? 0 : src_row) * kFp8SlotBytes + kFp8ScaleOff,
                            src_row < 0 ? 0u : 16u);
              }
            }
          }
          // The hardware arrives on the tile's full barrier for this thread
          // once all of this thread's copies so far have landed; the thread
          // itself never waits on them.
          cp_async_arrive_on(full);
        };
        // A barrier test sits in the memory pipe behind this warp's earlier
        // copies, so every wait costs about one drain of that queue.  With a
        // ring deeper than two blocks (N <= 32) the slots of a block are usually
        // all free already: test them together and issue every free tile back
        // to back, blocking only when none is free.  With the two-block ring of
        // N = 64 the slots free one by one behind P.V; there, waiting for each
        // tile in turn measures faster.
        if constexpr (N != 64) {
          uint32_t done = 0;
          while (done != 0x1fu) {
            uint32_t ready = 0;
#pragma unroll
            for (int step = 0; step < 5; ++step) {
              if (!((done >> step) & 1u)) {
                uint32_t empty, full, par, dst;
                int fc, nc;
                tile(step, empty, full, par, dst, fc, nc);
                if (mbar_test_wait(empty, par ^ 1u)) ready |= 1u << step;
              }
            }
            ready = __shfl_sync(0xffffffffu, ready, 0);
            if (ready == 0u) {
              const int step = __ffs(static_cast<int>(~done & 0x1fu)) - 1;
              uint32_t empty, full, par, dst;
              int fc, nc;
              tile(step, empty, full, par, dst, fc, nc);
              const bool ok = mbar_wait(empty, par ^ 1u, deadline, ab);
              if (!__all_sync(0xffffffffu, ok)) return false;
              ready = 1u << step;
            }
#pragma unroll
            for (int step = 0; step < 5; ++step) {
              if ((ready >> step) & 1u) {
                uint32_t empty, full, par, dst;
                int first_chunk, n_chunks;
                tile(step, empty, full, par, dst, first_chunk, n_chunks);
                copy_tile(step, full, dst, first_chunk, n_chunks);
              }
            }
            done |= ready;
          }
        } else {
          auto wait_and_copy = [&](int step) {
            uint32_t empty, full, par, dst;
            int first_chunk, n_chunks;
            tile(step, empty, full, par, dst, first_chunk, n_chunks);
            const bool ok = mbar_wait(empty, par ^ 1u, deadline, ab);
            if (!__all_sync(0xffffffffu, ok)) return false;
            copy_tile(step, full, dst, first_chunk, n_chunks);
            return true;
          };
          if constexpr (kFp8) {   // register-held codes: the step must be a constant
#pragma unroll
            for (int step = 0; step < 5; ++step)
              if (!wait_and_copy(step)) return false;
          } else {
#pragma unroll 1
            for (int step = 0; step < 5; ++step)
              if (!wait_and_copy(step)) return false;
          }
        }
        if constexpr (kFp8 && !kConv) {
          // This block's copies form one group; the previous block's group has
          // landed once at most this one is pending: convert that block.
          asm volatile("cp.async.commit_group;" ::: "memory");
          if (n > 0) {
            asm volatile("cp.async.wait_group 1;" ::: "memory");
            fp8_convert_block<L>(m, vbase, n - 1, warp, sel, piece, [](int, uint32_t) { return true; });
          }
        }
        ++n;
        ++ni;
      }
    }
    if constexpr (kCount) {
      // One add per item and head group 0 only (pieces of a cut unit add up).
      if (warp == 0 && lane == 0 && counted > 0 && item.unit % p.groups == 0) atomicAdd(p.valid_count + tok, counted);
      counted = 0;
      continue;
    }
    // End of the item: a marker the consumers take as "finish this unit".
    if (warp == 0) {
      const int k = ni % kInfoDepth;
      const bool ok = mbar_wait(smem_u32(&m.info_empty[k]), ((ni / kInfoDepth) & 1) ^ 1, deadline, ab);
      if (!__all_sync(0xffffffffu, ok)) return false;
      if (lane == 0) {
        m.info_blk[k] = -1;
        mbar_arrive(smem_u32(&m.info_full[k]));
      }
    }
    ++ni;
  }
  if constexpr (kFp8 && !kConv) {
    if (n > 0) {   // the last block's copies
      asm volatile("cp.async.wait_group 0;" ::: "memory");
      fp8_convert_block<L>(m, vbase, n - 1, warp, sel, piece, [](int, uint32_t) { return true; });
    }
  }
  return true;
}

// The index list is read from memory, or formed in place in the causal mode
// (decided once per launch, so the list walk carries no per-entry branch).
template <int N, bool kFp8>
__device__ __forceinline__ bool run_producer(const FwdParams& p, Misc& m, uint8_t* sbase) {
  if constexpr (kFp8)
    return run_producer_t<N, LayoutFor<N, kFp8>, Misc, false, false, false, true, (conv_warps<N, kFp8>() > 0)>(p, m, sbase);
  else
    return p.mode == kCausal ? run_producer_t<N, Layout<N>, Misc, false, true>(p, m, sbase)
                             : run_producer_t<N, Layout<N>, Misc, false, false>(p, m, sbase);
}

// ------------------------------------------------------------------ FP8 converters

// Converter warp cw (0..7) of the FP8 decode at 16 heads: follows the block
// sequence through the info ring like the consumers.  Warps 2u and 2u + 1
// take value tile u of every block (rows 0..31 and 32..63), so a block's four
// tiles are converted side by side as they land.  Per block a warp waits for
// its tile's raw codes in the value slot (raw_full), and for each half of its
// rows reads the codes (the slot's second chunk) and, once the whole warp
// has read them, rewrites those rows as bf16 code * 2^-120 (exact; the tile
// scales are applied by the softmax) in the 128B-swizzled layout the MMA
// descriptors read; then it arrives on the slot's full barrier.  A lane
// converts 16 codes of one row per row set; no other warp reads or writes
// these rows of the slot.
template <int N>
__device__ bool run_convert(const FwdParams& p, Misc& m, uint8_t* sbase, int cw) {
  using L = Layout<N, true>;
  constexpr int kPerTile = conv_warps<N, true>() / 4;   // converter warps per value tile
  static_assert(kPerTile * 4 == conv_warps<N, true>(), "converter warps: a multiple of four");
  constexpr int kPasses = kBlk / kPerTile / 16;          // passes of 16 rows per warp
  constexpr int kSets = 4;                               // row sets of 4 (8 lanes a row) per pass
  const volatile int* ab = &m.abort_flag;
  const uint32_t vbase = smem_u32(sbase + L::kVOff);
  const uint8_t* gbase = reinterpret_cast<const uint8_t*>(&m) - smem_u32(&m);   // generic address of shared offset 0
  const int lane = static_cast<int>(lane_id());
  const int sel = lane >> 3, piece = lane & 7;
  const int ch = piece >> 2, pc = (piece & 3) * 2;
  const int u = cw / kPerTile;                          // this warp's value tile
  const int row0 = (cw % kPerTile) * (kBlk / kPerTile); // and its rows
  int n = 0, ni = 0;
  ItemIter iter = items_begin(p);
  Item item;
  while (next_item(p, iter, item)) {
    const uint64_t deadline = global_timer_ns() + p.timeout_ns;   // every wait of this item is bounded from here
    for (;;) {
      const int k = ni % kInfoDepth;
      const bool ok = mbar_wait(smem_u32(&m.info_full[k]), (ni / kInfoDepth) & 1, deadline, ab);
      if (!__all_sync(0xffffffffu, ok)) return false;
      const int blk = *reinterpret_cast<volatile int32_t*>(&m.info_blk[k]);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&m.info_empty[k]));
      ++ni;
      if (blk < 0) break;
      const uint32_t vi = static_cast<uint32_t>(n) * 4u + static_cast<uint32_t>(u);
      const uint32_t sl = vi % L::kNV;
      const bool tok = mbar_wait(smem_u32(&m.raw_full[sl]), (vi / L::kNV) & 1u, deadline, ab);
      if (!__all_sync(0xffffffffu, tok)) return false;
      const uint32_t dst = vbase + sl * kPairBytes;
      const uint8_t* codes = gbase + dst + kChunkBytes;
#pragma unroll
      for (int pass = 0; pass < kPasses; ++pass) {
        uint4 c[kSets];
#pragma unroll
        for (int it = 0; it < kSets; ++it)
          c[it] = *reinterpret_cast<const uint4*>(codes + (row0 + pass * 16 + it * 4 + sel) * 128 + piece * 16);
        // every lane has read these rows' codes before any lane overwrites them
        __syncwarp();
#pragma unroll
        for (int it = 0; it < kSets; ++it) {
          const int row = row0 + pass * 16 + it * 4 + sel;
          // 16 codes: columns 128 u + 16 piece .. + 15 = chunk piece / 4, 8-column
          // pieces 2 (piece % 4) and 2 (piece % 4) + 1 of the row
          const uint32_t at = dst + ch * kChunkBytes + row * 128;
          st_shared_v4(at + ((pc ^ (row & 7)) << 4), e4m3x2_bf16x2_shifted<0>(c[it].x),
                       e4m3x2_bf16x2_shifted<1>(c[it].x), e4m3x2_bf16x2_shifted<0>(c[it].y),
                       e4m3x2_bf16x2_shifted<1>(c[it].y));
          st_shared_v4(at + (((pc + 1) ^ (row & 7)) << 4), e4m3x2_bf16x2_shifted<0>(c[it].z),
                       e4m3x2_bf16x2_shifted<1>(c[it].z), e4m3x2_bf16x2_shifted<0>(c[it].w),
                       e4m3x2_bf16x2_shifted<1>(c[it].w));
        }
      }
      // the tile's bf16 rows are written: order them before the tensor
      // core's reads (async proxy) and arrive on the slot's full barrier
      fence_proxy_async_smem();
      mbar_arrive(smem_u32(&m.v_full[sl]));
      ++n;
    }
  }
  return true;
}

// ------------------------------------------------------------------ MMA issuer

// The MMA work of a block is split between three issuing threads (one
// tcgen05 issuer sustains ~59 cycles per MMA here, several issuers more in
// aggregate), each with its own dependencies so none waits behind another:
//   QK part 0: QK^T over value pairs 0,1 and the rope columns
//   QK part 1: QK^T over value pairs 2,3
//   PV:        P.V for all of dv, as soon as the softmax has written P^T
// Each QK part accumulates its own partial S^T; the softmax adds the two.
// kRawCodes (FP8 at 16 heads): the value pairs hold the codes (times
// 2^-120); each pair (a 128-column scale tile) and the rope get a partial S^T
// of their own, at TMEM columns (5 (n & 1) + tile) N, tile 4 the rope.
template <int N, int PART, class L>
__device__ __forceinline__ bool issue_qk(Misc& m, uint32_t qbase, uint32_t vbase, uint32_t rbase, uint32_t tmem,
                                         int n, uint64_t deadline, const volatile int* ab) {
  constexpr uint32_t kIdescQK = idesc_bf16_f32(64, N, false, false);
  const uint32_t tS = tmem + static_cast<uint32_t>(PART * 2 + (n & 1)) * N;
  auto tile_acc = [&](int t) { return tmem + static_cast<uint32_t>(5 * (n & 1) + t) * N; };
  // Each tile's MMAs go as soon as that tile has landed (acquire, then a
  // proxy fence: the tiles were written by cp.async, the generic proxy, and
  // are read by the tensor core, the async proxy), so that only the last
  // tile's MMAs remain once the block's last copies land.
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int pr = 2 * PART + i;
    const uint32_t vi = static_cast<uint32_t>(n) * 4u + static_cast<uint32_t>(pr);
    const uint32_t slot = vi % L::kNV;
    if (!mbar_wait(smem_u32(&m.v_full[slot]), (vi / L::kNV) & 1u, deadline, ab)) return false;
    fence_proxy_async_smem();
    tc_fence_after();
#pragma unroll
    for (int c = 0; c < 2; ++c) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t a = smem_desc(vbase + slot * kPairBytes + c * kChunkBytes + kk * 32, 16, 1024, SWZ_128B);
        const uint64_t b = smem_desc(qbase + (2 * pr + c) * N * 128 + kk * 32, 16, 1024, SWZ_128B);
        if constexpr (L::kRawCodes)
          mma_bf16_ss(tile_acc(pr), a, b, kIdescQK, (c | kk) != 0 ? 1u : 0u);
        else
          mma_bf16_ss(tS, a, b, kIdescQK, (i | c | kk) != 0 ? 1u : 0u);
      }
    }
  }
  if (PART == 0) {
    const uint32_t rs = static_cast<uint32_t>(n) % L::kNR;
    if (!mbar_wait(smem_u32(&m.rp_full[rs]), (static_cast<uint32_t>(n) / L::kNR) & 1u, deadline, ab)) return false;
    fence_proxy_async_smem();
    tc_fence_after();
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const uint64_t a = smem_desc(rbase + rs * kChunkBytes + kk * 32, 16, 1024, SWZ_128B);
      const uint64_t b = smem_desc(qbase + 8 * N * 128 + kk * 32, 16, 1024, SWZ_128B);
      if constexpr (L::kRawCodes)
        mma_bf16_ss(tile_acc(4), a, b, kIdescQK, kk != 0 ? 1u : 0u);
      else
        mma_bf16_ss(tS, a, b, kIdescQK, 1u);
    }
  }
  mma_commit(smem_u32(&m.s_full[PART][n & 1]));
  return true;
}

template <int N, int PART, class L>
__device__ bool run_qk(const FwdParams& p, Misc& m, uint8_t* sbase, uint32_t tmem) {
  const volatile int* ab = &m.abort_flag;
  const uint32_t qbase = smem_u32(sbase + L::kQOff);
  const uint32_t vbase = smem_u32(sbase + L::kVOff);
  const uint32_t rbase = smem_u32(sbase + L::kROff);
  int n = 0, ni = 0, items = 0;   // blocks (S buffer parity), info entries, items
  ItemIter iter = items_begin(p);
  Item item;
  uint64_t deadline = 0;
  while (next_item(p, iter, item)) {
    deadline = global_timer_ns() + p.timeout_ns;   // every wait of this item is bounded from here
      // Q of this item, copied by the softmax warps (cp.async, generic proxy;
      // the tensor core reads it through the async proxy).
      if (!mbar_wait(smem_u32(&m.q_full), items & 1, deadline, ab)) return false;
      fence_proxy_async_smem();
      tc_fence_after();
      for (;;) {
        const int k = ni % kInfoDepth;
        if (!mbar_wait(smem_u32(&m.info_full[k]), (ni / kInfoDepth) & 1, deadline, ab)) return false;
        const int blk = *reinterpret_cast<volatile int32_t*>(&m.info_blk[k]);
        mbar_arrive(smem_u32(&m.info_empty[k]));
        ++ni;
        if (blk < 0) break;
        // S buffer n&1 was last read by the softmax of block n-2.
        if (n >= 2 && !mbar_wait(smem_u32(&m.p_full[n & 1]), ((n - 2) >> 1) & 1, deadline, ab)) return false;
        if (!issue_qk<N, PART, L>(m, qbase, vbase, rbase, tmem, n, deadline, ab)) return false;
        ++n;
      }
      // Q may be replaced once this thread's QK^T MMAs have completed.
      mma_commit(smem_u32(&m.q_empty));
      ++items;
  }
  return true;
}

// kRawCodes: V^T holds the codes (times 2^-120), and value tile mt contracts
// with its own scaled P^T tile (the rope slot's mt-th quarter).
template <int N, class L>
__device__ bool run_pv(const FwdParams& p, Misc& m, uint8_t* sbase, uint32_t tmem) {
  constexpr uint32_t kIdescPV = idesc_bf16_f32(128, N, true, true);
  constexpr uint32_t kPTile = L::kRawCodes ? kBlk * L::kPRow : 0;   // bytes between the scaled P^T tiles
  const volatile int* ab = &m.abort_flag;
  const uint32_t vbase = smem_u32(sbase + L::kVOff);
  const uint32_t rbase = smem_u32(sbase + L::kROff);
  const uint32_t tO = tmem + L::kOCol;
  int n = 0, ni = 0;   // blocks (ring positions), info entries
  ItemIter iter = items_begin(p);
  Item item;
  uint64_t deadline = 0;
  while (next_item(p, iter, item)) {
    deadline = global_timer_ns() + p.timeout_ns;   // every wait of this item is bounded from here
    int nl = 0;          // blocks of this item: the first one starts O^T afresh
    for (;; ++n, ++nl) {
      const int k = ni % kInfoDepth;
      if (!mbar_wait(smem_u32(&m.info_full[k]), (ni / kInfoDepth) & 1, deadline, ab)) return false;
      const int blk = *reinterpret_cast<volatile int32_t*>(&m.info_blk[k]);
      mbar_arrive(smem_u32(&m.info_empty[k]));
      ++ni;
      if (blk < 0) break;
      if (!mbar_wait(smem_u32(&m.p_full[n & 1]), (n >> 1) & 1, deadline, ab)) return false;
      tc_fence_after();
      const uint32_t rs = static_cast<uint32_t>(n) % L::kNR;
#pragma unroll 1
      for (int mt = 0; mt < 4; ++mt) {
        const uint32_t s = (static_cast<uint32_t>(n) * 4u + static_cast<uint32_t>(mt)) % L::kNV;
#pragma unroll
        for (int ks = 0; ks < kBlk / 16; ++ks) {
          const uint64_t a = smem_desc(vbase + s * kPairBytes + ks * 2048, kChunkBytes, 1024, SWZ_128B);
          const uint64_t b = smem_desc(rbase + rs * kChunkBytes + mt * kPTile + ks * 16 * L::kPRow,
                                       16 * L::kPRow * 8, 8 * L::kPRow, L::kPSwz);
          mma_bf16_ss(tO + mt * N, a, b, kIdescPV, (nl > 0 || ks > 0) ? 1u : 0u);
        }
        mma_commit(smem_u32(&m.v_empty[s]));
      }
      mma_commit(smem_u32(&m.rp_empty[rs]));
    }
    // O^T of an item that issued blocks is complete (the softmax waits on this
    // only for such items, so the two sides count the same phases).
    if (nl > 0) mma_commit(smem_u32(&m.o_full));
  }
  return true;
}

// ------------------------------------------------------------------ softmax + epilogue

// S^T row of this thread's half: HH consecutive heads starting at the
// half's first head (16x32bx2 read, upper half offset by HH columns).
// Merge of a unit that kBlockRanges cut between CTAs, for the heads [h_lo,
// h_hi) of one softmax group (128 threads): LSE = ln sum_s exp(LSE_s),
// out = sum_s exp(LSE_s - LSE) * O_s, each O_s already normalised over its
// piece (the LSE merge of the TileLang page's split-KV decode), taken in one
// pass over the pieces in order with a running maximum.  Sixteen threads
// share a (token, head) row, eight rows at a time; a thread owns the float4
// columns c16 + 16 k of the 512-wide row, so sixteen threads read 256
// contiguous bytes per load.  slots[s] is piece s's partial slot.  The
// partials were written by other CTAs: they are read from L2 (__ldcg) after
// the arrival count that made this the last piece.
__device__ void merge_unit(const FwdParams& p, int u, int h_lo, int h_hi, int tid, const int* slots, int pieces) {
  const int tok = u / p.groups;
  const int g64 = (u % p.groups) * 64;
  const int c16 = tid & 15;
  constexpr int kF4 = kDv / 4;   // float4 per row
  for (int h = h_lo + (tid >> 4); h < h_hi; h += 8) {
    float mrun = -INFINITY, l = 0.f;
    float4 acc[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 2
    for (int sp = 0; sp < pieces; ++sp) {
      const int slot = slots[sp];
      const float ls = __ldcg(p.part_lse + static_cast<size_t>(slot) * p.part_rows + h);
      const float4* src = reinterpret_cast<const float4*>(p.part_o) + (static_cast<size_t>(slot) * p.part_rows + h) * kF4 + c16;
      float4 v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = __ldcg(src + 16 * k);
      if (ls == -INFINITY) continue;   // an empty piece
      const float mn = fmaxf(mrun, ls);
      const float a = expf(mrun - mn), w = expf(ls - mn);
      l = l * a + w;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        acc[k].x = acc[k].x * a + w * v[k].x;
        acc[k].y = acc[k].y * a + w * v[k].y;
        acc[k].z = acc[k].z * a + w * v[k].z;
        acc[k].w = acc[k].w * a + w * v[k].w;
      }
      mrun = mn;
    }
    const int row = tok * p.h_q + g64 + h;
    const float inv = mrun == -INFINITY ? 0.f : 1.0f / l;
    if (c16 == 0) p.lse[row] = mrun == -INFINITY ? -INFINITY : mrun + logf(l);
    uint2* o = reinterpret_cast<uint2*>(p.out + static_cast<size_t>(row) * kDv) + c16;
#pragma unroll
    for (int k = 0; k < 8; ++k)
      o[16 * k] = make_uint2(pack_bf16x2(acc[k].x * inv, acc[k].y * inv), pack_bf16x2(acc[k].z * inv, acc[k].w * inv));
  }
}

// Pieces of unit u under kBlockRanges (1 when one CTA runs it whole).
__device__ __forceinline__ int unit_pieces(const FwdParams& p, int u) {
  const long long total = static_cast<long long>(p.n_tok) * p.groups * p.nb;
  const long long ub = static_cast<long long>(u) * p.nb;
  return range_cta(ub + p.nb - 1, total, p.ctas) - range_cta(ub, total, p.ctas) + 1;
}

template <int HH>
__device__ __forceinline__ void load_s_half(uint32_t taddr, float* v) {
  if constexpr (HH == 16) tmem_ld16x2_x16<16>(taddr, v);
  else tmem_ld16x2_x8<8>(taddr, v);
}

template <int N, class L>
__device__ bool run_softmax(const FwdParams& p, Misc& m, uint8_t* sbase, uint32_t tmem, int grp) {
  constexpr int H = L::kHG;            // heads this group owns (16 or 32)
  const volatile int* ab = &m.abort_flag;
  const uint32_t bar_id = 1u + static_cast<uint32_t>(grp);
  const int warp = static_cast<int>(threadIdx.x >> 5);
  const int lane = static_cast<int>(lane_id());
  const int tid = static_cast<int>(threadIdx.x) - softmax_warp0(grp) * 32;  // 0..127 within the group
  const int hb = grp * H;                              // first head of the group
  const int q4 = warp & 3;                             // TMEM lane quarter of this warp
  // The M=64 result sits in 16 lanes per quarter: both half-warps work on
  // the same 16 rows, the lower half on heads [hb, hb+H/2), the upper half on
  // [hb+H/2, hb+H).
  constexpr int HH = H / 2;
  const int hsub = (lane >> 4) * HH;                   // first head of this half, within the group
  const int row = q4 * 16 + (lane & 15);               // kv row of the block
  const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
  const uint32_t tO = tmem + lane_off + L::kOCol + hb;
  const uint32_t qbase = smem_u32(sbase + L::kQOff);
  const uint32_t rbase = smem_u32(sbase + L::kROff);

  int n = 0, ni = 0;        // blocks (buffer positions), info entries
  int items = 0, filled = 0; // items, items that issued blocks (o_full phases)
  ItemIter iter = items_begin(p);
  Item item;
  uint64_t deadline = 0;
  // Q rows of this group's heads for unit u -> shared memory, K-major with
  // the 128B swizzle, by cp.async so all loads are in flight at once; heads
  // past h_q are zero-filled.  The hardware arrives on q_full for this thread
  // once its copies have landed (the QK^T issuers fence the async proxy
  // after acquiring it), so no softmax thread waits on them.
  auto issue_q = [&](int u) {
    const int qtok = u / p.groups, qh0 = (u % p.groups) * 64;
    const int qhv = min(N, p.h_q - qh0);
    const __nv_bfloat16* qt = p.q + (static_cast<size_t>(qtok) * p.h_q + qh0) * kDqk;
    for (int x = tid; x < H * 72; x += 128) {
      const int h = hb + x / 72, rem = x % 72, c = rem >> 3, piece = rem & 7;
      const bool live = h < qhv;
      const __nv_bfloat16* src = qt + static_cast<size_t>(live ? h : 0) * kDqk + c * 64 + piece * 8;
      cp_async_16(qbase + c * (N * 128) + h * 128 + ((piece ^ (h & 7)) << 4), src, live ? 16u : 0u);
    }
    cp_async_arrive_on(smem_u32(&m.q_full));
  };
  bool q_issued = false;   // the current item's Q copies were issued during the previous item
  while (next_item(p, iter, item)) {
    deadline = global_timer_ns() + p.timeout_ns;   // every wait of this item is bounded from here
    const int tok = item.unit / p.groups;
    const int h0 = (item.unit % p.groups) * 64;
    const int hv = min(N, p.h_q - h0);
    if (!q_issued) issue_q(item.unit);   // the first item (later ones are issued ahead)
    q_issued = false;
    // (read after the first block's max barrier; the previous item's
    // epilogue, the last reader, has finished on this thread's side)
    if (tid < H) m.mrun[hb + tid] = -INFINITY;

    // Shares of the running sums of exp2(s - m), kept with the running max:
    // each block's row values go through the first two levels of the
    // half-warp butterfly (rows r, r ^ 4, r ^ 8, r ^ 12 of the quarter added),
    // so this thread holds heads hl0 .. hl0 + HH/4 - 1 of its four rows; the
    // rest of the butterfly runs once, at the end of the item.
    constexpr int HQ = HH / 4;
    const bool up8 = (lane & 8) != 0, up4 = (lane & 4) != 0;
    const int hl0 = hb + hsub + (up8 ? 2 * HQ : 0) + (up4 ? HQ : 0);
    float lpart[HQ];
#pragma unroll
    for (int i = 0; i < HQ; ++i) lpart[i] = 0.f;
    int nl = 0;   // blocks of this item
    for (;;) {
      const int k = ni % kInfoDepth;
      // Every wait is followed by a barrier that ORs the failures of the
      // group's 128 threads, so they all continue or all return together.
      const bool iok = mbar_wait(smem_u32(&m.info_full[k]), (ni / kInfoDepth) & 1, deadline, ab);
      ++ni;
      const int blk = iok ? *reinterpret_cast<volatile int32_t*>(&m.info_blk[k]) : -1;
      const uint32_t bits = *reinterpret_cast<volatile uint32_t*>(&m.info_mask[k][row & 1]);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&m.info_empty[k]));
      bool sok = true;
      if (blk >= 0) {
        sok = mbar_wait(smem_u32(&m.s_full[0][n & 1]), (n >> 1) & 1, deadline, ab) &&
              mbar_wait(smem_u32(&m.s_full[1][n & 1]), (n >> 1) & 1, deadline, ab);
        // kRawCodes: the block's tile scales landed with its rope tile (the
        // slot is not refilled before this block's P.V has completed)
        if constexpr (L::kRawCodes)
          sok = sok && mbar_wait(smem_u32(&m.rp_full[n % L::kNR]), (n / L::kNR) & 1, deadline, ab);
      }
      if (bar_red_or_128(bar_id, !(iok && sok))) return false;
      if (blk < 0) break;
      tc_fence_after();
      const bool valid = ((bits >> (row >> 1)) & 1u) != 0u;
      const uint32_t tSa = tmem + lane_off + static_cast<uint32_t>(n & 1) * N + hb;        // part 0
      const uint32_t tSb = tmem + lane_off + static_cast<uint32_t>(2 + (n & 1)) * N + hb;  // part 1
      // kRawCodes: the row's four tile scales
      float4 tsc = make_float4(0.f, 0.f, 0.f, 0.f);
      if constexpr (L::kRawCodes)
        tsc = *reinterpret_cast<const float4*>(sbase + L::kScOff + (n % L::kNR) * 1024 + row * 16);

      // The row's scaled scores (log2 units), masked rows -inf.
      auto load_scores = [&](float (&v)[HH]) {
        if constexpr (L::kRawCodes) {
          // S = sum over the value tiles of scale_t * (codes_t . q_t) + rope;
          // the partial sums hold codes_t . q_t times 2^-120 (taken back in
          // two factors, 2^56 with the scales and 2^64 on their sum)
          const uint32_t t0 = tmem + lane_off + static_cast<uint32_t>(5 * (n & 1)) * N + hb;
          float t[4][HH];
#pragma unroll
          for (int j = 0; j < 4; ++j) load_s_half<HH>(t0 + j * N, t[j]);
          load_s_half<HH>(t0 + 4 * N, v);
          tmem_wait_ld();
          const float sl = p.scale_log2 * 0x1p56f;
          const float a0 = tsc.x * sl, a1 = tsc.y * sl, a2 = tsc.z * sl, a3 = tsc.w * sl;
#pragma unroll
          for (int i = 0; i < HH; ++i)
            v[i] = valid ? v[i] * p.scale_log2 + (t[0][i] * a0 + t[1][i] * a1 + t[2][i] * a2 + t[3][i] * a3) * 0x1p64f
                         : -INFINITY;
        } else {
          float t[HH];
          load_s_half<HH>(tSa, v);
          load_s_half<HH>(tSb, t);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < HH; ++i) v[i] = valid ? (v[i] + t[i]) * p.scale_log2 : -INFINITY;
        }
      };
      float s[HH];
      load_scores(s);
      // The running maxima move only when a head's block max passes them by
      // more than 2^8 (lazy rescale), and always with the item's first block.
      // Any row can see that on its own: only then does the group reduce the
      // block max over the 64 rows and update the maxima.
      bool need = nl == 0;
#pragma unroll
      for (int i = 0; i < HH; ++i) need |= s[i] > m.mrun[hb + hsub + i] + kLazyRescale;
      if (bar_red_or_128(bar_id, need)) {
        // (the reduction consumes s; the scores are read again below)
        half_xreduce<HH, true>(s, lane, m.red[q4] + hb + hsub);
        named_bar_sync(bar_id, 128);
        bool grew = false;
        if (tid < H) {
          const int h = hb + tid;
          const float bm = fmaxf(fmaxf(m.red[0][h], m.red[1][h]), fmaxf(m.red[2][h], m.red[3][h]));
          const float mo = m.mrun[h];
          const float mn = (bm > mo + kLazyRescale) ? bm : mo;
          m.alpha[h] = fast_exp2(mo - mn);
          m.mrun[h] = mn;
          grew = (mn != mo);
        }
        const bool rescale = bar_red_or_128(bar_id, grew);
        if (nl > 0) {
#pragma unroll
          for (int i = 0; i < HQ; ++i) lpart[i] *= m.alpha[hl0 + i];
        }
        if (rescale && nl > 0) {
          // O^T must hold exactly the blocks before this one: wait for the
          // previous block's P.V (its last commits release that block's rope /
          // P^T slot), then rescale this group's head columns.
          const int pb = n - 1;
          const bool pok = mbar_wait(smem_u32(&m.rp_empty[pb % L::kNR]), (pb / L::kNR) & 1, deadline, ab);
          tc_fence_after();
          if (bar_red_or_128(bar_id, !pok)) return false;
#pragma unroll 1
          for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
            for (int g = 0; g < H / 16; ++g) {
              float o[16];
              tmem_ld16(tO + mt * N + g * 16, o);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 16; ++i) o[i] *= m.alpha[hb + g * 16 + i];
              tmem_st16(tO + mt * N + g * 16, o);
            }
          }
          tmem_wait_st();
        }
        load_scores(s);
      }
      // P^T row (bf16) into the rope slot of this block, MN-major swizzled,
      // and the row's shares of the sums.
      {
        const uint32_t prow = rbase + (n % L::kNR) * kChunkBytes + row * L::kPRow;
        const uint32_t sw = (static_cast<uint32_t>(row * L::kPRow) >> 7) & static_cast<uint32_t>(L::kPRow / 16 - 1);
#pragma unroll
        for (int c = 0; c < HH / 8; ++c) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int h = hb + hsub + c * 8 + i;
            s[c * 8 + i] = valid ? fast_exp2(s[c * 8 + i] - m.mrun[h]) : 0.f;
          }
          const uint32_t chunk = static_cast<uint32_t>((hb + hsub) / 8 + c);
          if constexpr (L::kRawCodes) {
            // value tile t's P^T: the row's P times its scale of tile t and
            // 2^88, bf16 (against codes times 2^-120: O^T holds out * 2^-32)
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const float f = (t == 0 ? tsc.x : (t == 1 ? tsc.y : (t == 2 ? tsc.z : tsc.w))) * 0x1p88f;
              st_shared_v4(prow + static_cast<uint32_t>(t * kBlk * L::kPRow) + ((chunk ^ sw) << 4),
                           pack_bf16x2(s[c * 8 + 0] * f, s[c * 8 + 1] * f), pack_bf16x2(s[c * 8 + 2] * f, s[c * 8 + 3] * f),
                           pack_bf16x2(s[c * 8 + 4] * f, s[c * 8 + 5] * f), pack_bf16x2(s[c * 8 + 6] * f, s[c * 8 + 7] * f));
            }
          } else {
            st_shared_v4(prow + ((chunk ^ sw) << 4), pack_bf16x2(s[c * 8 + 0], s[c * 8 + 1]),
                         pack_bf16x2(s[c * 8 + 2], s[c * 8 + 3]), pack_bf16x2(s[c * 8 + 4], s[c * 8 + 5]),
                         pack_bf16x2(s[c * 8 + 6], s[c * 8 + 7]));
          }
        }
        float h8[2 * HQ];
#pragma unroll
        for (int i = 0; i < 2 * HQ; ++i) {
          const float send = up8 ? s[i] : s[i + 2 * HQ];
          const float keep = up8 ? s[i + 2 * HQ] : s[i];
          h8[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
        }
#pragma unroll
        for (int i = 0; i < HQ; ++i) {
          const float send = up4 ? h8[i] : h8[i + HQ];
          const float keep = up4 ? h8[i + HQ] : h8[i];
          lpart[i] += keep + __shfl_xor_sync(0xffffffffu, send, 4);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(smem_u32(&m.p_full[n & 1]));
      ++n;
      ++nl;
    }
    // The item's sums over the 64 rows, per head (published by the barrier
    // after the o_full wait below).
    if (nl > 0) half_xreduce<HQ, false, 2>(lpart, lane, m.rsum[q4] + hl0);

    // The next item's Q, once this item's QK^T MMAs (the readers of Q) have
    // completed: its copies fly during this item's last P.V and epilogue,
    // which no longer touch the Q region, and the next item's QK^T can start
    // as soon as they land.
    {
      ItemIter peek = iter;
      Item nx;
      if (next_item(p, peek, nx)) {
        const bool qok = mbar_wait(smem_u32(&m.q_empty), items & 1, deadline, ab);
        if (bar_red_or_128(bar_id, !qok)) return false;
        issue_q(nx.unit);
        q_issued = true;
      }
    }

    // ---------------------------------------------------------- epilogue
    // O^T is complete once the P.V of the item's last block has; an item with
    // no block issued none (and P.V signals nothing for it).
    if (nl > 0) {
      const bool ook = mbar_wait(smem_u32(&m.o_full), filled & 1, deadline, ab);
      tc_fence_after();
      if (bar_red_or_128(bar_id, !ook)) return false;
      ++filled;
    }
    const size_t tok_h = static_cast<size_t>(tok) * p.h_q + h0;
    if (tid < H) {
      const int h = hb + tid;
      const float lrun = nl > 0 ? (m.rsum[0][h] + m.rsum[1][h]) + (m.rsum[2][h] + m.rsum[3][h]) : 0.f;
      float lse;
      if (nl > 0) {
        lse = (m.mrun[h] + log2f(lrun)) * 0.69314718055994530942f;
        m.fin[h] = (L::kRawCodes ? 0x1p32f : 1.0f) / lrun;   // kRawCodes: O^T holds out * 2^-32
      } else {
        lse = -INFINITY;
        m.fin[h] = 0.f;
      }
      if (h < hv) {
        if (item.slot >= 0) p.part_lse[static_cast<size_t>(item.slot) * p.part_rows + h] = lse;
        else p.lse[tok_h + h] = lse;
      }
    }
    named_bar_sync(bar_id, 128);
    const int dvrow = q4 * 32 + lane;   // O^T (M=128) lane of this thread
    // The group's normalisers in registers: read once here, not after every
    // store (which the compiler must assume may alias them).
    float fin[H];
#pragma unroll
    for (int i = 0; i < H; ++i) fin[i] = m.fin[hb + i];
    if (item.slot >= 0) {
      // fp32 partials: 32 consecutive dv per warp store (128 B), already coalesced.
      float* dst = p.part_o + (static_cast<size_t>(item.slot) * p.part_rows + hb) * kDv + dvrow;
#pragma unroll 1
      for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
        for (int g = 0; g < H / 16; ++g) {
          float o[16];
          if (nl > 0) {
            tmem_ld16(tO + mt * N + g * 16, o);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] = 0.f;
          }
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int hl = g * 16 + i;
            if (hb + hl < hv) dst[static_cast<size_t>(hl) * kDv + mt * 128] = o[i] * fin[hl];
          }
        }
      }
      // The piece is written (its LSEs by the owner threads above).  After
      // the group's barrier one thread counts the piece with a release add,
      // which publishes the group's writes; the group whose count completes
      // the unit acquires the others' and merges every piece into out / LSE
      // for its heads.
      named_bar_sync(bar_id, 128);
      if (tid < 32) {
        // lane 0 counts the piece; if it completes the unit, the warp lists
        // the pieces' slots (CTAs c_first .. c_last: slot 2c when the unit is
        // that CTA's first item, else 2c + 1)
        int last = 0;
        if (lane == 0)
          last = atomic_add_release_gpu(p.merge_count + item.unit * 2 + grp, 1) + 1 == unit_pieces(p, item.unit);
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
          fence_acquire_gpu();
          const long long total = static_cast<long long>(p.n_tok) * p.groups * p.nb;
          const long long ub = static_cast<long long>(item.unit) * p.nb;
          const int c_first = range_cta(ub, total, p.ctas);
          const int pieces = range_cta(ub + p.nb - 1, total, p.ctas) - c_first + 1;
          if (lane < pieces) {
            const int c = c_first + lane;
            m.merge_slot[grp][lane] = 2 * c + (range_start(c, total, p.ctas) < ub ? 1 : 0);
          }
          if (lane == 0) m.merge_pieces[grp] = pieces;
        } else if (lane == 0) {
          m.merge_pieces[grp] = 0;
        }
      }
      named_bar_sync(bar_id, 128);
      if (m.merge_pieces[grp] > 0)
        merge_unit(p, item.unit, hb, min(hb + H, hv), tid, m.merge_slot[grp], m.merge_pieces[grp]);
    } else {
      // bf16 output straight from TMEM: thread (q4, lane) holds dv = 128 mt +
      // 32 q4 + lane for each head; the lanes of an even/odd pair swap half
      // their heads so that each stores bf16x2 pairs (dv, dv + 1): a warp
      // store covers two 64-byte runs of two head rows.
      const bool odd = (lane & 1) != 0;
      __nv_bfloat16* orow = p.out + tok_h * kDv;
#pragma unroll 1
      for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
        for (int g = 0; g < H / 16; ++g) {
          float o[16];
          if (nl > 0) {
            tmem_ld16(tO + mt * N + g * 16, o);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] = 0.f;
          }
          const int dv0 = mt * 128 + q4 * 32 + (lane & ~1);
#pragma unroll
          for (int i = 0; i < 16; i += 2) {
            // even lane: head i with the odd lane's dv; odd lane: head i + 1 with the even lane's
            const float mine = odd ? o[i + 1] * fin[g * 16 + i + 1] : o[i] * fin[g * 16 + i];
            const float give = odd ? o[i] * fin[g * 16 + i] : o[i + 1] * fin[g * 16 + i + 1];
            const float got = __shfl_xor_sync(0xffffffffu, give, 1);
            const int hl = g * 16 + i + (odd ? 1 : 0);
            const uint32_t v = odd ? pack_bf16x2(got, mine) : pack_bf16x2(mine, got);
            if (hb + hl < hv) *reinterpret_cast<uint32_t*>(orow + static_cast<size_t>(hb + hl) * kDv + dv0) = v;
          }
        }
      }
    }
    ++items;
  }
  return true;
}

// ------------------------------------------------------------------ kernel

// kFp8: the FP8-cache instantiation (kPagedFp8); only the gather differs.
template <int N, bool kFp8 = false>
__global__ void __launch_bounds__(fwd_threads<N, kFp8>(), 1) sparse_mla_fwd_kernel(const __grid_constant__ FwdParams p) {
  using L = LayoutFor<N, kFp8>;
  constexpr int kConvWarps = conv_warps<N, kFp8>();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sbase = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Misc& m = *reinterpret_cast<Misc*>(sbase + L::kMiscOff);
  const int warp = static_cast<int>(threadIdx.x >> 5);
  const int lane = static_cast<int>(lane_id());

  // The producers' first reads (the first item's index window and, paged,
  // its request's page-table row) head a chain of dependent round trips:
  // start their lines into L2 while the CTA sets up.
  if (warp < kProducerWarps && p.mode != kCausal) {
    ItemIter it0 = items_begin(p);
    Item first;
    if (next_item(p, it0, first)) {
      const int tok = first.unit / p.groups;
      const int32_t* irow = p.indices + static_cast<size_t>(tok) * p.topk;
      const int e0 = first.jb * kBlk;
      const int e1 = min(p.topk, min(first.je, first.jb + 32) * kBlk);   // the first window of blocks
      for (int e = e0 + static_cast<int>(threadIdx.x) * 32; e < e1; e += kProducerWarps * 32 * 32)
        prefetch_line_l2(irow + e);
      if ((p.mode == kPaged || p.mode == kPagedFp8) && p.max_blocks > 0) {
        const int32_t* trow = p.block_table + static_cast<size_t>(tok / p.s_next) * p.max_blocks;
        for (int e = static_cast<int>(threadIdx.x) * 32; e < p.max_blocks; e += kProducerWarps * 32 * 32)
          prefetch_line_l2(trow + e);
      }
    }
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < L::kNV; ++i) {
      // the producer threads (cp.async), or the two converter warps of the tile
      mbar_init(smem_u32(&m.v_full[i]), kConvWarps > 0 ? 32 * kConvWarps / 4 : kProducerWarps * 32);   // converters: a tile's warps
      mbar_init(smem_u32(&m.v_empty[i]), 1);
    }
    for (int i = 0; i < (kConvWarps > 0 ? L::kNV : 0); ++i)
      mbar_init(smem_u32(&m.raw_full[i]), kProducerWarps * 32);   // producer threads (cp.async)
    for (int i = 0; i < L::kNR; ++i) {
      mbar_init(smem_u32(&m.rp_full[i]), kProducerWarps * 32);
      mbar_init(smem_u32(&m.rp_empty[i]), 1);
    }
    for (int i = 0; i < kInfoDepth; ++i) {
      mbar_init(smem_u32(&m.info_full[i]), 1);
      mbar_init(smem_u32(&m.info_empty[i]), 3 + 4 * L::kGroups + kConvWarps);
    }
    mbar_init(smem_u32(&m.q_full), 128 * L::kGroups);         // every softmax thread's Q copies (noinc)
    mbar_init(smem_u32(&m.q_empty), 2);                       // the two QK^T issuers
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&m.s_full[0][i]), 1);
      mbar_init(smem_u32(&m.s_full[1][i]), 1);
      mbar_init(smem_u32(&m.p_full[i]), 128 * L::kGroups);
    }
    for (int i = 0; i < 3; ++i) mbar_init(smem_u32(&m.drain[i]), 1);
    mbar_init(smem_u32(&m.cand_full), kProducerWarps);
    mbar_init(smem_u32(&m.o_full), 1);
    m.abort_flag = 0;
    m.prior_error = *reinterpret_cast<volatile int*>(&g_device_error);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&m.tmem_base), L::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = m.tmem_base;

  if (m.prior_error == 0) {
    if (warp < kProducerWarps) {
      if (!run_producer<N, kFp8>(p, m, sbase)) raise_error(m, kErrProducerWait);
      // Drain: every copy this thread issued has landed before the CTA can
      // exit, whether or not the consumers got to it.
      asm volatile("cp.async.wait_all;" ::: "memory");
    } else if (warp == kMmaWarp || warp == kMmaWarpB || warp == L::kPvWarp) {
      if (lane == 0) {
        const int role = warp == kMmaWarp ? 0 : (warp == kMmaWarpB ? 1 : 2);
        const bool ok = role == 0 ? run_qk<N, 0, L>(p, m, sbase, tmem)
                                  : (role == 1 ? run_qk<N, 1, L>(p, m, sbase, tmem) : run_pv<N, L>(p, m, sbase, tmem));
        if (!ok) raise_error(m, kErrMmaWait);
        // Drain: every MMA this thread issued completes before TMEM is freed.
        const int never = 0;
        mma_commit(smem_u32(&m.drain[role]));
        mbar_wait(smem_u32(&m.drain[role]), 0, global_timer_ns() + 100000000ull, &never);
      }
      __syncwarp();
    } else if (kConvWarps > 0 && warp > L::kPvWarp) {
      if constexpr (kConvWarps > 0) {
        if (!run_convert<N>(p, m, sbase, warp - L::kPvWarp - 1)) raise_error(m, kErrProducerWait);
      }
    } else {
      const int grp = warp >= softmax_warp0(1) ? 1 : 0;
      if (!run_softmax<N, L>(p, m, sbase, tmem, grp)) raise_error(m, kErrSoftmaxWait);
      // Drain: this thread's Q copies have landed before the CTA can exit.
      asm volatile("cp.async.wait_all;" ::: "memory");
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, L::kTmemCols);
}

// ------------------------------------------------------------------ helper kernels

// Debug export of the number of valid entries per token: the forward's own
// producer walk (its item schedule, window scan, block skips, row mapping and
// validity ballots) with the copies left out.  Four producer warps per CTA,
// the launch's item schedule; p.valid_count is zeroed before the launch.
__global__ void __launch_bounds__(kProducerWarps * 32, 1) valid_count_kernel(const __grid_constant__ FwdParams p) {
  __shared__ Misc m;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&m.cand_full), kProducerWarps);
    m.abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (!run_producer_t<16, Layout<16>, Misc, false, false, true>(p, m, reinterpret_cast<uint8_t*>(&m)))
    raise_error(m, kErrProducerWait);
}

// Every entry masked (no KV rows at all): out = 0, LSE = -inf.
__global__ void fill_masked_kernel(__nv_bfloat16* __restrict__ out, float* __restrict__ lse, long long n_th) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < n_th) lse[i] = -INFINITY;
  const long long n_el = n_th * kDv;
  for (long long e = i; e < n_el; e += static_cast<long long>(gridDim.x) * blockDim.x)
    out[e] = __float2bfloat16_rn(0.f);
}

}  // namespace smla
