// DSA sparse-MLA attention backward for sm_103a (cp.async gather + tcgen05).
//
// Gradients of the forward (fwd_kernel.cuh) with respect to q and kv for an
// upstream gradient dout of out; the LSE output carries no gradient.  This is
// the backward the training users pair with the forward (prime-rl page:
// forward and backward sparse-attention timings).  Per token t, head h and
// the token's valid gathered rows K (V = K[:, :512], the same latent rows):
//
//   P  = exp(sm_scale q K^T - LSE)          (LSE from the forward)
//   dP = dout V^T,   D = rowsum(dout * out)
//   dS = P (dP - D)
//   dq_t          = sm_scale dS K
//   dkv[r]       += sm_scale dS^T q_t      (all 576 columns)
//   dkv[r, :512] += P^T dout_t
//
// Work decomposition: the forward's persistent grid and gather (the same
// producer), with units of one token x up to 16 heads (U = 1) or, above 16
// heads, one token x up to 32 heads taken as two halves of 16 (U = 2): each
// block's dKV then sums both halves before it is drained, so the gather and
// the dkv reductions (the L2 traffic that bounds the backward) are paid once
// per 32 heads.  Per 64-row block:
//
//   warps 0..3   producers: gather the block's rows (value pairs + rope tile)
//                and publish its 64 row ids.
//   warps 4, 9   S^T = K Q^T and dP^T = V dout^T (swap-AB, M = 64 kv rows,
//                N = every head of the unit) into TMEM: with U = 1 each
//                takes half of the value pairs (warp 4 also the rope columns
//                of S); with U = 2 warp 4 issues S and warp 9 dP, each over
//                all pairs at N = 32 (Q and dout of the 32 heads form one
//                K-major tile per 64-dim chunk).
//   warps 5..8   P, dS from S, dP, the LSE and D; write P^T and
//                (sm_scale dS)^T of every half as bf16 rows into shared
//                memory.
//   warp 10      dQ^T += K^T (sm_scale dS)^T over all heads of the unit (K^T
//                the MN-major view of the gathered tile, as V^T in the
//                forward's P.V; accumulated in TMEM over the unit), which frees the block's
//                tiles; then the block's dKV rows in column chunks taken
//                in turn by two TMEM buffers, one chunk's MMAs overlapping
//                the other's drain (128 x 4 and 64 with U = 1; 128, 64, 128,
//                64, 128, 64 with U = 2):
//                dKV = sum over halves of (sm_scale dS)^T Q + P^T [dout, 0]
//                (M = 64 rows, K = 16 heads per half, Q and dout read as
//                MN-major B operands).
//   warps 11..14 drain each dKV chunk from TMEM and add it into dkv (fp32)
//                with 16-byte reductions, by the block's row ids, two lanes
//                per aligned 32-byte sector in each instruction.
//
// At the end of a unit the softmax warps write dq (fp32) from TMEM.  All
// waits are bounded like the forward's.
#pragma once
#include "fwd_kernel.cuh"

namespace smla {

constexpr int kBwdHeads = 16;   // heads per half: the N of the S / dP / dQ MMAs

template <int U>
struct BwdLayout {
  static constexpr int N = kBwdHeads;
  static constexpr int H = U * N;                       // heads per unit
  static constexpr int kNV = U == 1 ? 9 : 6;            // value ring: 2.25 / 1.5 blocks
  static constexpr int kNR = U == 1 ? 3 : 2;            // rope ring
  static constexpr int kPRow = N * 2;                   // bytes of one P^T / dS^T row
  static constexpr uint32_t kPSwz = SWZ_32B;
  static constexpr int kPSBytes = kBlk * kPRow;         // one P^T or dS^T tile of one half (2 KB)
  static constexpr int kPSLbo = 2 * kPSBytes;           // dS^T of half 1 from that of half 0 ([half][P^T, dS^T])
  // Q and dout: 64-dim chunks of all H heads of the unit (128 B per head,
  // K-major with the 128B swizzle), so that the S, dP and dQ MMAs take every
  // head of the unit at once (N = H); half h is rows [16 h, 16 h + 16).
  static constexpr int kQChunk = H * 128;
  static constexpr int kQOff = 0;
  static constexpr int kDOOff = kQOff + 9 * kQChunk;
  static constexpr int kVOff = kDOOff + 8 * kQChunk;
  static constexpr int kROff = kVOff + kNV * kPairBytes;
  static constexpr int kPSOff = kROff + kNR * kChunkBytes;   // [buffer][half][P^T, dS^T]
  static constexpr int kMiscOff = kPSOff + 2 * U * 2 * kPSBytes;
  // TMEM columns
  static constexpr int kTS = 0;                         // S^T: U = 1 [part][buffer] x 16; U = 2 [buffer] x 32
  static constexpr int kTdP = 4 * N;                    // dP^T: the same
  static constexpr int kTdQ = 8 * N;                    // dQ^T: four M=128 tiles of 128 dims, the M=64 rope tile; H columns each
  static constexpr int kTdKV = U == 1 ? 256 : kTdQ + 5 * H;   // dKV chunk buffers (M=64)
  // dKV column chunks in two TMEM buffers taken in turn (buffer b of the
  // CTA's chunk g is g % 2), so that one chunk's MMAs run while the other
  // buffer drains.  U = 1: five chunks (128 x 4, 64), two 128-column
  // buffers; U = 2: six chunks (128, 64, 128, 64, 128, 64), a 128- and a
  // 64-column buffer.  Chunks start on 64-dim boundaries (the MN-major
  // Q / dout swizzle atoms).
  static constexpr int kKVChunks = U == 1 ? 5 : 6;
  static constexpr int kKVBufs = 2;
  __device__ static constexpr int kv_col0(int c) { return U == 1 ? c * 128 : (c >> 1) * 192 + (c & 1) * 128; }
  __device__ static constexpr int kv_width(int c) { return U == 1 ? (c < 4 ? 128 : 64) : ((c & 1) ? 64 : 128); }
  __device__ static constexpr int kv_tmem(int b) { return kTdKV + b * 128; }
  static constexpr int kTmemCols = 512;
  // warp roles
  static constexpr int kQkWarp0 = 4, kSoftWarp0 = 5, kQkWarp1 = 9, kGradWarp = 10, kDrainWarp0 = 11;
  static constexpr int kThreads = 15 * 32;
};
static_assert(BwdLayout<1>::kTdQ + 5 * BwdLayout<1>::N <= BwdLayout<1>::kTdKV, "TMEM map");
static_assert(BwdLayout<1>::kTdKV + 128 + 128 <= BwdLayout<1>::kTmemCols, "TMEM map");
static_assert(BwdLayout<2>::kTdKV + 128 + 64 <= BwdLayout<2>::kTmemCols, "TMEM map");
static_assert(BwdLayout<1>::kVOff % 1024 == 0 && BwdLayout<1>::kROff % 1024 == 0 && BwdLayout<1>::kPSOff % 1024 == 0,
              "swizzled tiles start on 1024-byte boundaries");
static_assert(BwdLayout<2>::kVOff % 1024 == 0 && BwdLayout<2>::kROff % 1024 == 0 && BwdLayout<2>::kPSOff % 1024 == 0,
              "swizzled tiles start on 1024-byte boundaries");

template <int U>
struct __align__(16) BwdMisc {
  uint64_t v_full[BwdLayout<U>::kNV], v_empty[BwdLayout<U>::kNV];
  uint64_t rp_full[BwdLayout<U>::kNR], rp_empty[BwdLayout<U>::kNR];
  uint64_t info_full[kInfoDepth], info_empty[kInfoDepth];
  uint64_t q_full, q_empty, s_full[2][2], pds_full[2], pds_empty[2], dkv_full[2], dkv_empty[2], dq_full,
      drain[3],
      cand_full;
  int32_t info_blk[kInfoDepth];
  uint32_t info_mask[kInfoDepth][2];
  int32_t info_rows[kInfoDepth][kBlk];
  uint32_t cand[2][kProducerWarps];
  float dsum[U * kBwdHeads];   // D = rowsum(dout * out) per head of the unit
  float lse2[U * kBwdHeads];   // LSE * log2(e)
  uint32_t tmem_base;
  int abort_flag;
  int prior_error;
};

template <int U>
constexpr int bwd_smem_bytes() { return BwdLayout<U>::kMiscOff + static_cast<int>(sizeof(BwdMisc<U>)) + 1024; }
static_assert(bwd_smem_bytes<1>() <= kMaxSmem, "smem budget (backward)");
static_assert(bwd_smem_bytes<2>() <= kMaxSmem, "smem budget (backward, 32-head units)");

enum BwdErrCode : int { kErrBwdGradWait = 0x401, kErrBwdDrainWait = 0x501 };

__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

template <int U>
__device__ __forceinline__ void bwd_raise(BwdMisc<U>& m, int code) {
  *reinterpret_cast<volatile int*>(&m.abort_flag) = 1;
  atomicCAS(&g_device_error, 0, code);
}

// ------------------------------------------------------------------ S, dP issuers

// S^T (QK^T) and dP^T of block n for one part.  U = 1: value pairs 2P and
// 2P+1 (part 0 also the rope columns of S), the two parts summed by the
// softmax.  U = 2: part 0 issues S^T and part 1 dP^T, each over every value
// pair (S also the rope) and all 32 heads in one N = 32 MMA per k-step.  The
// A operand (the gathered rows, K-major) is shared by the two products; B is
// Q for S and dout for dP.
template <int U, int PART>
__device__ __forceinline__ bool bwd_issue_s_dp(BwdMisc<U>& m, uint32_t qbase, uint32_t dobase, uint32_t vbase,
                                               uint32_t rbase, uint32_t tmem, int n, uint64_t deadline,
                                               const volatile int* ab) {
  using L = BwdLayout<U>;
  constexpr int NM = L::H;                        // MMA N: every head of the unit
  constexpr int kPairs = U == 1 ? 2 : 4;          // value pairs this issuer takes
  constexpr int kPair0 = U == 1 ? 2 * PART : 0;
  constexpr bool kS = U == 1 || PART == 0;        // issues S^T
  constexpr bool kDP = U == 1 || PART == 1;       // issues dP^T
  constexpr bool kRope = PART == 0;
  constexpr uint32_t kIdesc = idesc_bf16_f32(64, NM, false, false);
  const uint32_t buf = U == 1 ? static_cast<uint32_t>(PART * 2 + (n & 1)) : static_cast<uint32_t>(n & 1);
  const uint32_t tS = tmem + static_cast<uint32_t>(L::kTS) + buf * NM;
  const uint32_t tP = tmem + static_cast<uint32_t>(L::kTdP) + buf * NM;
  uint32_t slot[kPairs];
#pragma unroll
  for (int i = 0; i < kPairs; ++i) {
    const uint32_t vi = static_cast<uint32_t>(n) * 4u + static_cast<uint32_t>(kPair0 + i);
    slot[i] = vi % L::kNV;
    if (!mbar_wait(smem_u32(&m.v_full[slot[i]]), (vi / L::kNV) & 1u, deadline, ab)) return false;
  }
  const uint32_t rs = static_cast<uint32_t>(n) % L::kNR;
  if (kRope && !mbar_wait(smem_u32(&m.rp_full[rs]), (static_cast<uint32_t>(n) / L::kNR) & 1u, deadline, ab))
    return false;
  fence_proxy_async_smem();
  tc_fence_after();
#pragma unroll
  for (int i = 0; i < kPairs; ++i) {
    const int pr = kPair0 + i;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t a = smem_desc(vbase + slot[i] * kPairBytes + c * kChunkBytes + kk * 32, 16, 1024, SWZ_128B);
        const uint32_t acc = (i | c | kk) != 0 ? 1u : 0u;
        if (kS) mma_bf16_ss(tS, a, smem_desc(qbase + (2 * pr + c) * L::kQChunk + kk * 32, 16, 1024, SWZ_128B), kIdesc, acc);
        if (kDP)
          mma_bf16_ss(tP, a, smem_desc(dobase + (2 * pr + c) * L::kQChunk + kk * 32, 16, 1024, SWZ_128B), kIdesc, acc);
      }
    }
  }
  if (kRope) {
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const uint64_t a = smem_desc(rbase + rs * kChunkBytes + kk * 32, 16, 1024, SWZ_128B);
      const uint64_t b = smem_desc(qbase + 8 * L::kQChunk + kk * 32, 16, 1024, SWZ_128B);
      mma_bf16_ss(tS, a, b, kIdesc, 1u);
    }
  }
  mma_commit(smem_u32(&m.s_full[PART][n & 1]));
  return true;
}

template <int U, int PART>
__device__ bool run_bwd_s_dp(const FwdParams& p, BwdMisc<U>& m, uint8_t* sbase, uint32_t tmem) {
  using L = BwdLayout<U>;
  const volatile int* ab = &m.abort_flag;
  const uint32_t qbase = smem_u32(sbase + L::kQOff);
  const uint32_t dobase = smem_u32(sbase + L::kDOOff);
  const uint32_t vbase = smem_u32(sbase + L::kVOff);
  const uint32_t rbase = smem_u32(sbase + L::kROff);
  int n = 0, ni = 0, items = 0;
  ItemIter iter = items_begin(p);
  Item item;
  uint64_t deadline = 0;
  while (next_item(p, iter, item)) {
    deadline = global_timer_ns() + p.timeout_ns;
    if (!mbar_wait(smem_u32(&m.q_full), items & 1, deadline, ab)) return false;   // Q and dout of this unit
    tc_fence_after();
    for (;;) {
      const int k = ni % kInfoDepth;
      if (!mbar_wait(smem_u32(&m.info_full[k]), (ni / kInfoDepth) & 1, deadline, ab)) return false;
      const int blk = *reinterpret_cast<volatile int32_t*>(&m.info_blk[k]);
      mbar_arrive(smem_u32(&m.info_empty[k]));
      ++ni;
      if (blk < 0) break;
      // S / dP buffer n&1 was last read by the softmax of block n-2.
      if (n >= 2 && !mbar_wait(smem_u32(&m.pds_full[n & 1]), ((n - 2) >> 1) & 1, deadline, ab)) return false;
      if (!bwd_issue_s_dp<U, PART>(m, qbase, dobase, vbase, rbase, tmem, n, deadline, ab)) return false;
      ++n;
    }
    mma_commit(smem_u32(&m.q_empty));   // Q / dout may be replaced once these MMAs complete
    ++items;
  }
  return true;
}

// ------------------------------------------------------------------ dQ, dKV issuer

template <int U>
__device__ bool run_bwd_grad(const FwdParams& p, BwdMisc<U>& m, uint8_t* sbase, uint32_t tmem) {
  using L = BwdLayout<U>;
  constexpr int N = L::N;
  constexpr int NM = L::H;                           // MMA N of dQ: every head of the unit
  constexpr uint32_t kIdescDQ = idesc_bf16_f32(128, NM, true, true);
  constexpr uint32_t kIdescDQr = idesc_bf16_f32(64, NM, true, true);
  const volatile int* ab = &m.abort_flag;
  const uint32_t qbase = smem_u32(sbase + L::kQOff);
  const uint32_t dobase = smem_u32(sbase + L::kDOOff);
  const uint32_t vbase = smem_u32(sbase + L::kVOff);
  const uint32_t rbase = smem_u32(sbase + L::kROff);
  const uint32_t psbase = smem_u32(sbase + L::kPSOff);
  const uint32_t tdQ = tmem + L::kTdQ;
  int n = 0, ni = 0, chunks = 0;
  ItemIter iter = items_begin(p);
  Item item;
  uint64_t deadline = 0;
  while (next_item(p, iter, item)) {
    deadline = global_timer_ns() + p.timeout_ns;
    int nl = 0;
    for (;; ++n, ++nl) {
      const int k = ni % kInfoDepth;
      if (!mbar_wait(smem_u32(&m.info_full[k]), (ni / kInfoDepth) & 1, deadline, ab)) return false;
      const int blk = *reinterpret_cast<volatile int32_t*>(&m.info_blk[k]);
      mbar_arrive(smem_u32(&m.info_empty[k]));
      ++ni;
      if (blk < 0) break;
      if (!mbar_wait(smem_u32(&m.pds_full[n & 1]), (n >> 1) & 1, deadline, ab)) return false;
      tc_fence_after();
      // this block's tiles: [half][P^T, dS^T]
      const uint32_t ps = psbase + static_cast<uint32_t>(n & 1) * static_cast<uint32_t>(U * 2 * L::kPSBytes);
      // dQ^T[576 x H] += K^T[576 x 64] dS^T[64 x H]: four 128-dim tiles of
      // the value pairs, then the 64 rope dims (M = 64).  B is MN-major over
      // the heads: with U = 2 the dS^T tiles of the two halves are its two
      // 16-head swizzle atoms, kLBO apart.  Each pair tile is free after its
      // MMAs (dP already used it; dKV does not read it).
      const uint32_t pds = ps + static_cast<uint32_t>(L::kPSBytes);   // dS^T of half 0
#pragma unroll 1
      for (int u = 0; u < 4; ++u) {
        const uint32_t s = (static_cast<uint32_t>(n) * 4u + static_cast<uint32_t>(u)) % L::kNV;
#pragma unroll
        for (int ks = 0; ks < kBlk / 16; ++ks) {
          const uint64_t a = smem_desc(vbase + s * kPairBytes + ks * 2048, kChunkBytes, 1024, SWZ_128B);
          const uint64_t b = smem_desc(pds + ks * 16 * L::kPRow, L::kPSLbo, 8 * L::kPRow, L::kPSwz);
          mma_bf16_ss(tdQ + u * NM, a, b, kIdescDQ, (nl > 0 || ks > 0) ? 1u : 0u);
        }
        mma_commit(smem_u32(&m.v_empty[s]));
      }
      const uint32_t rs = static_cast<uint32_t>(n) % L::kNR;
#pragma unroll
      for (int ks = 0; ks < kBlk / 16; ++ks) {
        const uint64_t a = smem_desc(rbase + rs * kChunkBytes + ks * 2048, kChunkBytes, 1024, SWZ_128B);
        const uint64_t b = smem_desc(pds + ks * 16 * L::kPRow, L::kPSLbo, 8 * L::kPRow, L::kPSwz);
        mma_bf16_ss(tdQ + 4 * NM, a, b, kIdescDQr, (nl > 0 || ks > 0) ? 1u : 0u);
      }
      mma_commit(smem_u32(&m.rp_empty[rs]));
      // dKV rows of the block in column chunks: the sum over halves of
      // (sm_scale dS)^T Q plus P^T [dout, 0].  A: the P^T / dS^T tiles as
      // K-major [64 rows x 16 heads]; B: the half's 16 rows of Q / dout as
      // MN-major [16 heads x dims] (their 64-dim chunks sit kQChunk bytes
      // apart).
#pragma unroll
      for (int c = 0; c < L::kKVChunks; ++c) {
        const int col0 = L::kv_col0(c);
        const int wq = L::kv_width(c);                                    // Q columns of the chunk
        const int wd = 512 - col0 < wq ? (512 - col0 > 0 ? 512 - col0 : 0) : wq;   // dout columns (may be none)
        const int b = chunks % L::kKVBufs;
        const uint32_t use = static_cast<uint32_t>(chunks / L::kKVBufs);
        const uint32_t tKV = tmem + static_cast<uint32_t>(L::kv_tmem(b));
        if (!mbar_wait(smem_u32(&m.dkv_empty[b]), (use & 1u) ^ 1u, deadline, ab)) return false;
        tc_fence_after();
#pragma unroll
        for (int h = 0; h < U; ++h) {
          const uint32_t pt = ps + static_cast<uint32_t>(h * 2) * L::kPSBytes;
          const uint64_t a_p = smem_desc(pt, 16, 8 * L::kPRow, L::kPSwz);
          const uint64_t a_ds = smem_desc(pt + L::kPSBytes, 16, 8 * L::kPRow, L::kPSwz);
          const uint64_t bq =
              smem_desc(qbase + h * N * 128 + (col0 / 64) * L::kQChunk, L::kQChunk, 1024, SWZ_128B);
          mma_bf16_ss(tKV, a_ds, bq, idesc_bf16_f32(64, wq, false, true), h > 0 ? 1u : 0u);
          if (wd > 0) {
            const uint64_t bd =
                smem_desc(dobase + h * N * 128 + (col0 / 64) * L::kQChunk, L::kQChunk, 1024, SWZ_128B);
            mma_bf16_ss(tKV, a_p, bd, idesc_bf16_f32(64, wd, false, true), 1u);
          }
        }
        mma_commit(smem_u32(&m.dkv_full[b]));
        ++chunks;
      }
      mma_commit(smem_u32(&m.pds_empty[n & 1]));
    }
    if (nl > 0) mma_commit(smem_u32(&m.dq_full));
    mma_commit(smem_u32(&m.q_empty));
  }
  return true;
}

// ------------------------------------------------------------------ dKV drain

// The block's rows over 64 columns: eight 16x32bx2.x4 reads with the half
// split at 4 columns, so threads l and l + 16 (the same row r = 16 q4 + l)
// hold columns [c, c + 4) and [c + 4, c + 8) of each 8-column step.  Their
// two 16-byte reductions then fill one aligned 32-byte sector in the same
// instruction (16 full sectors per instruction rather than 32 half ones:
// the L2 reduction traffic that bounds the backward is counted in sectors).
__device__ __forceinline__ void drain_load64(uint32_t taddr, int col, float* v) {
#pragma unroll
  for (int k = 0; k < 8; ++k) tmem_ld16x2_x4<4>(taddr + static_cast<uint32_t>(col + 8 * k), v + 4 * k);
}

__device__ __forceinline__ void drain_red64(const float* v, float* dst_row, int col, bool live, int half) {
  if (live) {
#pragma unroll
    for (int k = 0; k < 8; ++k)
      red_add_v4(dst_row + col + 8 * k + 4 * half, v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
  }
}

// One dKV chunk of w columns (a multiple of 64) into dkv, software-pipelined:
// the next 64 columns' TMEM reads are in flight while the current ones'
// reductions issue, so a chunk pays one TMEM round trip, not one per batch
// (the drain of the 16-head units: c2 bwd 1732 -> 1678 us).
__device__ __forceinline__ void drain_chunk(uint32_t taddr, int w, float* dst_row, bool live, int half) {
  float va[32], vb[32];
  drain_load64(taddr, 0, va);
  tmem_wait_ld();
#pragma unroll 1
  for (int col = 0; col < w; col += 128) {
    if (col + 64 < w) drain_load64(taddr, col + 64, vb);
    drain_red64(va, dst_row, col, live, half);
    tmem_wait_ld();
    if (col + 64 < w) {
      if (col + 128 < w) drain_load64(taddr, col + 128, va);
      drain_red64(vb, dst_row, col + 64, live, half);
      tmem_wait_ld();
    }
  }
}

// 32 columns of the block's rows, one TMEM round trip (the drain of the
// 32-head units: there the pipelined drain's burstier reductions measured
// slower, 25.5 against 22.9 ms at 8192 tokens x 64 heads).
__device__ __forceinline__ void drain_cols32(uint32_t taddr, int col, float* dst_row, bool live, int half) {
  float v[16];
#pragma unroll
  for (int k = 0; k < 4; ++k) tmem_ld16x2_x4<4>(taddr + static_cast<uint32_t>(col + 8 * k), v + 4 * k);
  tmem_wait_ld();
  if (live) {
#pragma unroll
    for (int k = 0; k < 4; ++k)
      red_add_v4(dst_row + col + 8 * k + 4 * half, v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
  }
}

template <int U>
__device__ bool run_bwd_drain(const FwdParams& p, BwdMisc<U>& m, uint32_t tmem) {
  using L = BwdLayout<U>;
  const volatile int* ab = &m.abort_flag;
  const int warp = static_cast<int>(threadIdx.x >> 5);
  const int lane = static_cast<int>(lane_id());
  const int q4 = warp & 3;
  const int r = q4 * 16 + (lane & 15);        // block row of this thread (M=64 layout)
  const int half = lane >> 4;
  const uint32_t tl = tmem + (static_cast<uint32_t>(q4 * 32) << 16);   // this warp's TMEM lanes
  int ni = 0, chunks = 0;
  ItemIter iter = items_begin(p);
  Item item;
  uint64_t deadline = 0;
  while (next_item(p, iter, item)) {
    deadline = global_timer_ns() + p.timeout_ns;
    for (;;) {
      const int k = ni % kInfoDepth;
      const bool iok = mbar_wait(smem_u32(&m.info_full[k]), (ni / kInfoDepth) & 1, deadline, ab);
      if (!__all_sync(0xffffffffu, iok)) return false;
      ++ni;
      const int blk = *reinterpret_cast<volatile int32_t*>(&m.info_blk[k]);
      const int row = blk < 0 ? -1 : *reinterpret_cast<volatile int32_t*>(&m.info_rows[k][r]);
      if (blk < 0) {
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&m.info_empty[k]));
        break;
      }
      float* dst = p.dkv + static_cast<size_t>(row < 0 ? 0 : row) * kDqk;
#pragma unroll 1
      for (int c = 0; c < L::kKVChunks; ++c) {
        const int b = chunks % L::kKVBufs;
        const uint32_t use = static_cast<uint32_t>(chunks / L::kKVBufs);
        const bool ok = mbar_wait(smem_u32(&m.dkv_full[b]), use & 1u, deadline, ab);
        if (!__all_sync(0xffffffffu, ok)) return false;
        tc_fence_after();
        const int col0 = L::kv_col0(c);
        const int w = L::kv_width(c);
        const uint32_t tKV = tl + static_cast<uint32_t>(L::kv_tmem(b));
        if constexpr (U == 1) {
          drain_chunk(tKV, w, dst + col0, row >= 0, half);
        } else {
#pragma unroll 1
          for (int col = 0; col < w; col += 32) drain_cols32(tKV, col, dst + col0, row >= 0, half);
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&m.dkv_empty[b]));
        ++chunks;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&m.info_empty[k]));   // row ids no longer needed
    }
  }
  return true;
}

// ------------------------------------------------------------------ P, dS and dq

template <int U>
__device__ bool run_bwd_softmax(const FwdParams& p, BwdMisc<U>& m, uint8_t* sbase, uint32_t tmem) {
  using L = BwdLayout<U>;
  constexpr int N = L::N;
  constexpr int H = L::H;                              // heads per unit
  constexpr int HH = N / 2;                            // heads per half-warp (of one half)
  const volatile int* ab = &m.abort_flag;
  constexpr uint32_t bar_id = 1u;
  const int warp = static_cast<int>(threadIdx.x >> 5);
  const int lane = static_cast<int>(lane_id());
  const int tid = static_cast<int>(threadIdx.x) - L::kSoftWarp0 * 32;   // 0..127
  const int q4 = warp & 3;
  const int hsub = (lane >> 4) * HH;
  const int row = q4 * 16 + (lane & 15);
  const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
  const uint32_t qbase = smem_u32(sbase + L::kQOff);
  const uint32_t dobase = smem_u32(sbase + L::kDOOff);
  const uint32_t psbase = smem_u32(sbase + L::kPSOff);
  const float sm_scale = p.sm_scale;
  int n = 0, ni = 0, items = 0, filled = 0;
  ItemIter iter = items_begin(p);
  Item item;
  uint64_t deadline = 0;
  while (next_item(p, iter, item)) {
    deadline = global_timer_ns() + p.timeout_ns;
    const int tok = item.unit / p.groups;
    const int h0 = (item.unit % p.groups) * H;
    const int hv = min(H, p.h_q - h0);
    const size_t tok_h = static_cast<size_t>(tok) * p.h_q + h0;
    if (items > 0) {
      // Q and dout are replaced once the previous unit's MMAs reading them
      // (S, dP and dKV) have completed.
      const bool ok = mbar_wait(smem_u32(&m.q_empty), (items - 1) & 1, deadline, ab);
      if (bar_red_or_128(bar_id, !ok)) return false;
    }
    // Q (9 chunks) and dout (8 chunks) of the unit's heads -> shared memory,
    // K-major with the 128B swizzle, all H heads per chunk; heads past h_q
    // are zero-filled.
    {
      const __nv_bfloat16* qt = p.q + tok_h * kDqk;
      for (int x = tid; x < H * 72; x += 128) {
        const int hd = x / 72, rem = x % 72, c = rem >> 3, piece = rem & 7;
        const bool live = hd < hv;
        cp_async_16(qbase + c * L::kQChunk + hd * 128 + ((piece ^ (hd & 7)) << 4),
                    qt + static_cast<size_t>(live ? hd : 0) * kDqk + c * 64 + piece * 8, live ? 16u : 0u);
      }
      const __nv_bfloat16* dt = p.dout + tok_h * kDv;
      for (int x = tid; x < H * 64; x += 128) {
        const int hd = x / 64, rem = x % 64, c = rem >> 3, piece = rem & 7;
        const bool live = hd < hv;
        cp_async_16(dobase + c * L::kQChunk + hd * 128 + ((piece ^ (hd & 7)) << 4),
                    dt + static_cast<size_t>(live ? hd : 0) * kDv + c * 64 + piece * 8, live ? 16u : 0u);
      }
      // D = rowsum(dout * out) per head: eight threads per head, 64 columns each.
      for (int h = tid >> 3; h < H; h += 16) {
        const int part = tid & 7;
        float acc = 0.f;
        if (h < hv) {
          const uint4* o4 = reinterpret_cast<const uint4*>(p.out + (tok_h + h) * kDv + part * 64);
          const uint4* d4 = reinterpret_cast<const uint4*>(p.dout + (tok_h + h) * kDv + part * 64);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint4 a = __ldg(o4 + i), b = __ldg(d4 + i);
            const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
            const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float2 fa = __bfloat1622float2(a2[j]), fb = __bfloat1622float2(b2[j]);
              acc += fa.x * fb.x + fa.y * fb.y;
            }
          }
        }
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        acc += __shfl_xor_sync(0xffffffffu, acc, 2);
        acc += __shfl_xor_sync(0xffffffffu, acc, 4);
        if (part == 0) {
          m.dsum[h] = acc;
          m.lse2[h] = h < hv ? __ldg(p.lse + tok_h + h) * 1.4426950408889634f : 0.f;
        }
      }
      asm volatile("cp.async.wait_all;" ::: "memory");
      fence_proxy_async_smem();
      named_bar_sync(bar_id, 128);
      if (tid == 0) mbar_arrive(smem_u32(&m.q_full));
    }
    float dsum[U][HH], lse2[U][HH];
#pragma unroll
    for (int hf = 0; hf < U; ++hf)
#pragma unroll
      for (int i = 0; i < HH; ++i) {
        dsum[hf][i] = m.dsum[hf * N + hsub + i];
        lse2[hf][i] = m.lse2[hf * N + hsub + i];
      }

    int nl = 0;
    for (;;) {
      const int k = ni % kInfoDepth;
      const bool iok = mbar_wait(smem_u32(&m.info_full[k]), (ni / kInfoDepth) & 1, deadline, ab);
      ++ni;
      if (bar_red_or_128(bar_id, !iok)) return false;
      const int blk = *reinterpret_cast<volatile int32_t*>(&m.info_blk[k]);
      const uint32_t bits = *reinterpret_cast<volatile uint32_t*>(&m.info_mask[k][row & 1]);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&m.info_empty[k]));
      if (blk < 0) break;
      const bool valid = ((bits >> (row >> 1)) & 1u) != 0u;
      // The P^T / dS^T buffer n&1 was last read by the dKV MMAs of block n-2.
      bool ok = n < 2 || mbar_wait(smem_u32(&m.pds_empty[n & 1]), ((n - 2) >> 1) & 1, deadline, ab);
      ok = ok && mbar_wait(smem_u32(&m.s_full[0][n & 1]), (n >> 1) & 1, deadline, ab) &&
           mbar_wait(smem_u32(&m.s_full[1][n & 1]), (n >> 1) & 1, deadline, ab);
      tc_fence_after();
      if (bar_red_or_128(bar_id, !ok)) return false;
      const uint32_t col = static_cast<uint32_t>(n & 1) * N;
      const uint32_t ps0 = psbase + static_cast<uint32_t>(n & 1) * static_cast<uint32_t>(U * 2 * L::kPSBytes);
      const uint32_t sw = (static_cast<uint32_t>(row * L::kPRow) >> 7) & static_cast<uint32_t>(L::kPRow / 16 - 1);
      const uint32_t off = static_cast<uint32_t>(row * L::kPRow) + (((static_cast<uint32_t>(hsub / 8)) ^ sw) << 4);
#pragma unroll
      for (int hf = 0; hf < U; ++hf) {
        // U = 1: S and dP are the sums of the two parts; U = 2: half hf's own.
        float s[HH], d[HH];
        if constexpr (U == 1) {
          float sb[HH], db[HH];
          tmem_ld16x2_x8<HH>(tmem + lane_off + L::kTS + col, s);
          tmem_ld16x2_x8<HH>(tmem + lane_off + L::kTS + 2 * N + col, sb);
          tmem_ld16x2_x8<HH>(tmem + lane_off + L::kTdP + col, d);
          tmem_ld16x2_x8<HH>(tmem + lane_off + L::kTdP + 2 * N + col, db);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < HH; ++i) {
            s[i] += sb[i];
            d[i] += db[i];
          }
        } else {
          tmem_ld16x2_x8<HH>(tmem + lane_off + L::kTS + 2 * col + hf * N, s);
          tmem_ld16x2_x8<HH>(tmem + lane_off + L::kTdP + 2 * col + hf * N, d);
          tmem_wait_ld();
        }
        float pr[HH], ds[HH];
#pragma unroll
        for (int i = 0; i < HH; ++i) {
          pr[i] = valid ? fast_exp2(s[i] * p.scale_log2 - lse2[hf][i]) : 0.f;
          ds[i] = pr[i] * (d[i] - dsum[hf][i]) * sm_scale;
        }
        const uint32_t ps = ps0 + static_cast<uint32_t>(hf * 2) * L::kPSBytes;
        st_shared_v4(ps + off, pack_bf16x2(pr[0], pr[1]), pack_bf16x2(pr[2], pr[3]), pack_bf16x2(pr[4], pr[5]),
                     pack_bf16x2(pr[6], pr[7]));
        st_shared_v4(ps + L::kPSBytes + off, pack_bf16x2(ds[0], ds[1]), pack_bf16x2(ds[2], ds[3]),
                     pack_bf16x2(ds[4], ds[5]), pack_bf16x2(ds[6], ds[7]));
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(smem_u32(&m.pds_full[n & 1]));
      ++n;
      ++nl;
    }

    // dq of the unit (fp32): dQ^T is complete once the dQ MMAs of its last
    // block have; a unit without blocks gets zeros.
    if (nl > 0) {
      const bool ok = mbar_wait(smem_u32(&m.dq_full), filled & 1, deadline, ab);
      tc_fence_after();
      if (bar_red_or_128(bar_id, !ok)) return false;
      ++filled;
    }
#pragma unroll 1
    for (int hf = 0; hf < U; ++hf) {
      float* dq = p.dq + (tok_h + hf * N) * kDqk;
      const int hvf = hv - hf * N;   // live heads of this half (may be <= 0)
#pragma unroll 1
      for (int mt = 0; mt < 5; ++mt) {
        float o[16];
        if (nl > 0) {
          tmem_ld16(tmem + lane_off + L::kTdQ + mt * H + hf * N, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) o[i] = 0.f;
        }
        // tiles 0..3: lane = dim 128 mt + 32 q4 + lane; the rope tile (M=64):
        // dims 512 + 16 q4 + lane for lanes 0..15.
        const int dim = mt < 4 ? mt * 128 + q4 * 32 + lane : 512 + q4 * 16 + lane;
        if (mt < 4 || lane < 16) {
#pragma unroll
          for (int h = 0; h < 16; ++h)
            if (h < hvf) dq[static_cast<size_t>(h) * kDqk + dim] = o[h];
        }
      }
    }
    tc_fence_before();
    ++items;
  }
  return true;
}

// ------------------------------------------------------------------ kernel

template <int U>
__global__ void __launch_bounds__(BwdLayout<U>::kThreads, 1) sparse_mla_bwd_kernel(const __grid_constant__ FwdParams p) {
  using L = BwdLayout<U>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sbase = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  BwdMisc<U>& m = *reinterpret_cast<BwdMisc<U>*>(sbase + L::kMiscOff);
  const int warp = static_cast<int>(threadIdx.x >> 5);
  const int lane = static_cast<int>(lane_id());

  if (threadIdx.x == 0) {
    for (int i = 0; i < L::kNV; ++i) {
      mbar_init(smem_u32(&m.v_full[i]), kProducerWarps * 32);
      mbar_init(smem_u32(&m.v_empty[i]), 1);
    }
    for (int i = 0; i < L::kNR; ++i) {
      mbar_init(smem_u32(&m.rp_full[i]), kProducerWarps * 32);
      mbar_init(smem_u32(&m.rp_empty[i]), 1);
    }
    for (int i = 0; i < kInfoDepth; ++i) {
      mbar_init(smem_u32(&m.info_full[i]), 1);
      mbar_init(smem_u32(&m.info_empty[i]), 3 + 4 + 4);   // two S/dP issuers, grad issuer, softmax and drain warps
    }
    mbar_init(smem_u32(&m.q_full), 1);
    mbar_init(smem_u32(&m.q_empty), 3);                   // both S/dP issuers and the grad issuer
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&m.s_full[0][i]), 1);
      mbar_init(smem_u32(&m.s_full[1][i]), 1);
      mbar_init(smem_u32(&m.pds_full[i]), 128);
      mbar_init(smem_u32(&m.pds_empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&m.dkv_full[i]), 1);
      mbar_init(smem_u32(&m.dkv_empty[i]), 128);
    }
    mbar_init(smem_u32(&m.dq_full), 1);
    for (int i = 0; i < 3; ++i) mbar_init(smem_u32(&m.drain[i]), 1);
    mbar_init(smem_u32(&m.cand_full), kProducerWarps);
    m.abort_flag = 0;
    m.prior_error = *reinterpret_cast<volatile int*>(&g_device_error);
    fence_mbar_init();
  }
  if (warp == L::kQkWarp0) {
    tmem_alloc(smem_u32(&m.tmem_base), L::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = m.tmem_base;

  if (m.prior_error == 0) {
    if (warp < kProducerWarps) {
      // The ring of U = 2 is 1.5 blocks deep: take its slots one by one (the
      // producer's strategy for shallow rings).
      if (!run_producer_t<U == 1 ? kBwdHeads : 64, L, BwdMisc<U>, true>(p, m, sbase)) bwd_raise(m, kErrProducerWait);
      asm volatile("cp.async.wait_all;" ::: "memory");
    } else if (warp == L::kQkWarp0 || warp == L::kQkWarp1 || warp == L::kGradWarp) {
      if (lane == 0) {
        const int role = warp == L::kQkWarp0 ? 0 : (warp == L::kQkWarp1 ? 1 : 2);
        const bool ok = role == 0 ? run_bwd_s_dp<U, 0>(p, m, sbase, tmem)
                                  : (role == 1 ? run_bwd_s_dp<U, 1>(p, m, sbase, tmem) : run_bwd_grad<U>(p, m, sbase, tmem));
        if (!ok) bwd_raise(m, role == 2 ? kErrBwdGradWait : kErrMmaWait);
        const int never = 0;
        mma_commit(smem_u32(&m.drain[role]));
        mbar_wait(smem_u32(&m.drain[role]), 0, global_timer_ns() + 100000000ull, &never);
      }
      __syncwarp();
    } else if (warp >= L::kDrainWarp0) {
      if (!run_bwd_drain<U>(p, m, tmem)) bwd_raise(m, kErrBwdDrainWait);
    } else {
      if (!run_bwd_softmax<U>(p, m, sbase, tmem)) bwd_raise(m, kErrSoftmaxWait);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == L::kQkWarp0) tmem_dealloc(tmem, L::kTmemCols);
}

}  // namespace smla
