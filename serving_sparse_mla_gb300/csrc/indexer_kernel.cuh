// DSA indexer scores and top-k selection for sm_103a (TMA + tcgen05).
//
// The step upstream of the sparse-MLA forward that produces its index
// lists.  The pages name the indexer and its top-k ("[Feature] Add optional
// FlashMLA backend for DSA Sparse MLA", Changes; "feat: add XTuner TileLang
// sparse MLA backend", Summary and Copilot overview) without printing the
// score formula; it is taken here as the DSA lightning indexer published
// with DeepSeek-V3.2:
//
//   I[t,s] = sum_j w[t,j] * relu(q[t,j,:] . k[s,:])       (j < H_I, width 128)
//
// over the positions s query t may see (the s_q queries of a sequence are
// the last s_q of its s_kv positions; for a paged decode cache, the s_next
// MTP rows of a request are its last s_next positions and its keys are read
// page by page through the block table).  A row's list holds the topk visible
// positions of largest score, equal scores ranked by position (smaller
// first), written in increasing position order and padded with -1; a row
// that sees at most topk positions takes all of them and is never scored.
//
// dsa_scores_kernel<H_I>: a dense contraction, so it runs on the tensor
// cores.  A work item is a group of G = 256 / H_I consecutive query rows
// (N = 256 columns: every head of every row) against up to 32 tiles of 128
// positions of their sequence (M = 128; fewer per item when a launch has
// few groups, so that every SM gets several items):
//
//   S^T[128 x 256] = K_tile[128 x 128] . Q_group^T[128 x 256]    (fp32, TMEM)
//
//   warp 0      TMA: per item the group's Q (two 32 KB boxes, 128B swizzle)
//               and its head weights (1-D bulk copy), then the K tiles (two
//               16 KB boxes each; four 8 KB boxes, two pages, for a paged
//               cache) through a 4-deep ring that runs ahead across items.
//   warp 1      one thread issues a tile's 8 MMAs (K = 16 each) into one of
//               two 256-column TMEM accumulators and commits.
//   warps 2..9  epilogue over half of the group's (row, head) columns each:
//               four threads share a position, each with 16 heads of it
//               (16x256b TMEM reads; the heads' weights stay in registers
//               for the item), relu and weights in packed fp32 FMAs, a
//               3-shuffle transpose-reduce to one score per thread, fp32
//               stores into the rows' logits (32 lanes: 32 consecutive
//               positions).  The accumulator is freed once read.
//
// A persistent grid (at most one CTA per SM, ~212 KB of shared memory each)
// walks items c, c + G, ... (dealt chunk by chunk, largest groups first);
// while an item runs, its successor's Q is prefetched into L2.  Rows that see at most `skip_len` positions
// get no tiles.  A group that straddles sequences is run as one segment per
// sequence, each against that sequence's keys.
//
// dsa_topk_kernel: one CTA per query row (256 threads; 1024 when rows pass
// 8192 positions).  The row's order-preserving
// integer keys (the image of fp32) are staged in shared memory when they
// fit; a radix select of the topk largest then counts digits of 11, 11 and
// 10 bits in shared-memory histograms (each pass over the keys still in
// the threshold class, stopping as soon as the class is taken whole), and
// an ordered compaction writes the selected positions in increasing order,
// taking equal scores at the threshold by position.
//
// All waits of the scores kernel are bounded like the forward's; a CTA that
// times out records an error, waits (bounded) for its copies and MMAs in
// flight, frees TMEM and returns.
#pragma once
#include <cuda.h>

#include "fwd_kernel.cuh"

namespace smla {

constexpr int kIdxD = 128;            // indexer head width
constexpr int kIdxTile = 128;         // positions per K tile (the MMA's M)
constexpr int kIdxN = 256;            // (row, head) columns of a group (the MMA's N)
constexpr int kIdxChunkTiles = 32;    // most tiles per item (4096 positions); a launch may take fewer
constexpr int kIdxStages = 4;
constexpr int kIdxMaxBatch = 2048;    // sequences whose offsets sit in shared memory
constexpr int kIdxEpiWarp0 = 2;
constexpr int kIdxThreads = 10 * 32;
constexpr int kIdxTmemCols = 512;

constexpr int kIdxQHalf = kIdxN * 128;                        // 256 rows x 64 columns (bf16)
constexpr int kIdxKHalf = kIdxTile * 128;                     // 128 rows x 64 columns
constexpr int kIdxKStage = 2 * kIdxKHalf;
constexpr int kIdxQOff = 0;
constexpr int kIdxKOff = kIdxQOff + 2 * kIdxQHalf;
constexpr int kIdxWOff = kIdxKOff + kIdxStages * kIdxKStage;  // head weights [2][256] fp32
constexpr int kIdxCuOff = kIdxWOff + 2 * kIdxN * 4;           // cu_q, cu_kv [kIdxMaxBatch + 1] each
constexpr int kIdxMiscOff = kIdxCuOff + ((2 * (kIdxMaxBatch + 1) * 4 + 15) / 16) * 16;

struct __align__(16) IdxMisc {
  uint64_t q_full, q_empty, k_full[kIdxStages], k_empty[kIdxStages], acc_full[2], acc_empty[2], w_full[2],
      w_empty[2], drain;
  uint32_t tmem_base;
  int abort_flag;
  int prior_error;
  int32_t pages[2 * kIdxChunkTiles];   // paged cache: the producer's current segment's page ids
};

constexpr int idx_smem_bytes() { return kIdxMiscOff + static_cast<int>(sizeof(IdxMisc)) + 1024; }
static_assert(idx_smem_bytes() <= kMaxSmem, "smem budget (indexer scores)");
static_assert(kIdxKOff % 1024 == 0 && kIdxKStage % 1024 == 0 && kIdxQHalf % 1024 == 0, "swizzled tiles");

enum IdxErrCode : int {
  kErrIdxProducerWait = 0x601,
  kErrIdxMmaWait = 0x602,
  kErrIdxEpilogueWait = 0x603,
  kErrIdxRowTooLong = 0x611,   // a sequence sees more positions than a logits row holds
};

constexpr int kIdxPage = 64;          // positions per page of a paged key cache

struct IdxParams {
  CUtensorMap map_q;          // bf16 [total_q * h_idx, 128]: box {64, 256}, 128B swizzle
  CUtensorMap map_k;          // bf16 [total_kv, 128]: box {64, 128}, 128B swizzle (paged: box {64, 64})
  const float* weights;       // [total_q, h_idx]
  const int32_t* cu_q;        // [batch + 1], null for one dense sequence or a paged cache
  const int32_t* cu_kv;
  const int32_t* block_table; // paged cache: [batch, max_blocks] pages of kIdxPage positions, else null
  const int32_t* seqlens;     // paged cache: [batch] positions per request
  int s_next, max_blocks, num_blocks;   // paged cache: query rows per request (the last s_next positions)
  float* scores;              // [n_rows, row_stride]: row r - row0 holds row r's positions
  long long row_stride;
  int total_q, total_kv, batch, h_idx;
  int row0, n_rows;           // the query rows of this launch
  int skip_len;               // rows seeing <= skip_len positions are not scored
  int groups;                 // ceil(n_rows / G)
  int kv_chunks;              // ceil(longest KV sequence / (128 chunk_tiles))
  int chunk_tiles;            // tiles per item, at most kIdxChunkTiles
  unsigned long long timeout_ns;
};

__device__ __forceinline__ void idx_raise(IdxMisc& m, int code) {
  *reinterpret_cast<volatile int*>(&m.abort_flag) = 1;
  atomicCAS(&g_device_error, 0, code);
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
               : "memory");
}

// (c0, c1) += (a0 * b0, a1 * b1): one packed fp32 FMA, each lane rounded
// as fmaf.
__device__ __forceinline__ void ffma2(float& c0, float& c1, float a0, float a1, float b0, float b1) {
  asm("{\n\t.reg .b64 pa, pb, pc;\n\t"
      "mov.b64 pa, {%2, %3};\n\t"
      "mov.b64 pb, {%4, %5};\n\t"
      "mov.b64 pc, {%0, %1};\n\t"
      "fma.rn.f32x2 pc, pa, pb, pc;\n\t"
      "mov.b64 {%0, %1}, pc;\n\t}"
      : "+f"(c0), "+f"(c1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// 4-byte asynchronous copy global -> shared (zero-filled when src_bytes is 0).
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

// Positions row r of sequence b sees: the sequence's queries are the last
// lq of its lk positions.
__device__ __forceinline__ int idx_visible(const int32_t* cq, const int32_t* ck, int b, int r) {
  const int lq = cq[b + 1] - cq[b], lk = ck[b + 1] - ck[b];
  const int v = r - cq[b] + lk - lq + 1;
  return v < 0 ? 0 : (v > lk ? lk : v);
}

// Last b in [0, batch) with cq[b] <= r.
__device__ __forceinline__ int idx_seq_of(const int32_t* cq, int batch, int r) {
  int lo = 0, hi = batch - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cq[mid] <= r) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// One run of a group's rows inside one sequence, with the tiles of the
// item's chunk it needs (t0 == t1: none).
struct IdxSeg {
  int b, r_begin, r_end, kv_begin, t0, t1;
};

// The segments of item (group g, chunk c), in row order.  Every role walks
// the same sequence.
struct IdxWalk {
  int r_first, r_stop, r, b, c;
  // Items are dealt chunk by chunk (every group's first 4096 positions,
  // then every group's next 4096, ...), and within a chunk the last groups
  // first: with causal rows the later groups see more positions, so every
  // CTA's share runs from large items to small and no CTA collects only
  // the short chunks.
  __device__ __forceinline__ void start(const IdxParams& p, const int32_t* cq, long long item) {
    const int g = p.groups - 1 - static_cast<int>(item % p.groups);
    c = static_cast<int>(item / p.groups);
    const int G = kIdxN / p.h_idx;
    r_first = p.row0 + g * G;
    const int end = p.row0 + p.n_rows;
    r_stop = r_first + G < end ? r_first + G : end;
    r = r_first;
    b = idx_seq_of(cq, p.batch, r_first);
  }
  __device__ __forceinline__ bool next(const IdxParams& p, const int32_t* cq, const int32_t* ck, IdxSeg& s) {
    while (r < r_stop && b < p.batch) {
      const int e = r_stop < cq[b + 1] ? r_stop : cq[b + 1];
      if (e > r) {
        s.b = b;
        s.r_begin = r;
        s.r_end = e;
        s.kv_begin = ck[b];
        long long v = idx_visible(cq, ck, b, e - 1);   // the segment's longest row
        if (v > p.row_stride) v = p.row_stride;
        s.t0 = s.t1 = c * p.chunk_tiles;
        if (v > p.skip_len) {
          const int nt = static_cast<int>((v + kIdxTile - 1) / kIdxTile);
          s.t1 = nt < s.t0 + p.chunk_tiles ? nt : s.t0 + p.chunk_tiles;
          if (s.t1 < s.t0) s.t1 = s.t0;
        }
        r = e;
        ++b;
        return true;
      }
      ++b;
    }
    return false;
  }
};

// ------------------------------------------------------------------ roles

__device__ __forceinline__ bool idx_producer(const IdxParams& p, IdxMisc& m, uint32_t sb, const int32_t* cq,
                                             const int32_t* ck, uint32_t& kcount, uint32_t& qcount,
                                             uint32_t& wcount) {
  const volatile int* ab = &m.abort_flag;
  const long long n_items = static_cast<long long>(p.groups) * p.kv_chunks;
  for (long long it = blockIdx.x; it < n_items; it += gridDim.x) {
    const uint64_t deadline = global_timer_ns() + p.timeout_ns;
    IdxWalk w;
    w.start(p, cq, it);
    IdxSeg s;
    bool first = true;
    while (w.next(p, cq, ck, s)) {
      if (p.block_table != nullptr && s.t1 > s.t0) {
        // The segment's page ids, all in flight at once (one round trip
        // rather than one per tile); ids past the table read as -1.
        const int32_t* bt = p.block_table + static_cast<size_t>(s.b) * p.max_blocks;
        const int lp0 = 2 * s.t0, npg = 2 * (s.t1 - s.t0);
        for (int i = 0; i < npg; ++i) {
          if (lp0 + i < p.max_blocks) cp_async_4(smem_u32(&m.pages[i]), bt + lp0 + i, 4u);
          else m.pages[i] = -1;
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
      }
      for (int t = s.t0; t < s.t1; ++t) {
        if (first) {
          first = false;
          // the group's Q, once the previous item's MMAs have read it
          if (!mbar_wait(smem_u32(&m.q_empty), (qcount & 1u) ^ 1u, deadline, ab)) return false;
          mbar_arrive_expect_tx(smem_u32(&m.q_full), 2 * kIdxQHalf);
          const int y = w.r_first * p.h_idx;
          tma_load_2d(sb + kIdxQOff, &p.map_q, 0, y, smem_u32(&m.q_full));
          tma_load_2d(sb + kIdxQOff + kIdxQHalf, &p.map_q, 64, y, smem_u32(&m.q_full));
          ++qcount;
          // the next item's Q into L2, so its load after this item's MMAs is short
          if (it + gridDim.x < n_items) {
            IdxWalk nx;
            nx.start(p, cq, it + gridDim.x);
            if (nx.r_first != w.r_first) {
              tma_prefetch_2d(&p.map_q, 0, nx.r_first * p.h_idx);
              tma_prefetch_2d(&p.map_q, 64, nx.r_first * p.h_idx);
            }
          }
          // its head weights, into the buffer the epilogue released
          const uint32_t wb = wcount & 1u;
          if (!mbar_wait(smem_u32(&m.w_empty[wb]), ((wcount >> 1) & 1u) ^ 1u, deadline, ab)) return false;
          const uint32_t bytes = static_cast<uint32_t>((w.r_stop - w.r_first) * p.h_idx) * 4u;
          mbar_arrive_expect_tx(smem_u32(&m.w_full[wb]), bytes);
          bulk_load(sb + kIdxWOff + wb * kIdxN * 4, p.weights + static_cast<long long>(w.r_first) * p.h_idx, bytes,
                    smem_u32(&m.w_full[wb]));
          ++wcount;
        }
        const uint32_t slot = kcount % kIdxStages;
        if (!mbar_wait(smem_u32(&m.k_empty[slot]), ((kcount / kIdxStages) & 1u) ^ 1u, deadline, ab)) return false;
        mbar_arrive_expect_tx(smem_u32(&m.k_full[slot]), kIdxKStage);
        const uint32_t dst = sb + kIdxKOff + slot * kIdxKStage;
        if (p.block_table == nullptr) {
          const int y = s.kv_begin + t * kIdxTile;
          tma_load_2d(dst, &p.map_k, 0, y, smem_u32(&m.k_full[slot]));
          tma_load_2d(dst + kIdxKHalf, &p.map_k, 64, y, smem_u32(&m.k_full[slot]));
        } else {
          // Two pages per tile, each a 64-row box per column half; a page id
          // outside the table or the pool reads as zeros.
#pragma unroll
          for (int pg = 0; pg < 2; ++pg) {
            const int blk = m.pages[2 * (t - s.t0) + pg];
            const int y = blk >= 0 && blk < p.num_blocks ? blk * kIdxPage : -kIdxPage;
            const uint32_t d = dst + static_cast<uint32_t>(pg * kIdxPage * 128);
            tma_load_2d(d, &p.map_k, 0, y, smem_u32(&m.k_full[slot]));
            tma_load_2d(d + kIdxKHalf, &p.map_k, 64, y, smem_u32(&m.k_full[slot]));
          }
        }
        ++kcount;
      }
    }
  }
  return true;
}

__device__ __forceinline__ bool idx_mma(const IdxParams& p, IdxMisc& m, uint32_t sb, uint32_t tmem,
                                        const int32_t* cq, const int32_t* ck) {
  constexpr uint32_t kIdesc = idesc_bf16_f32(kIdxTile, kIdxN, false, false);
  const volatile int* ab = &m.abort_flag;
  uint32_t kcount = 0, acount = 0, qcount = 0;
  const long long n_items = static_cast<long long>(p.groups) * p.kv_chunks;
  for (long long it = blockIdx.x; it < n_items; it += gridDim.x) {
    const uint64_t deadline = global_timer_ns() + p.timeout_ns;
    IdxWalk w;
    w.start(p, cq, it);
    IdxSeg s;
    bool q_ready = false;
    while (w.next(p, cq, ck, s)) {
      for (int t = s.t0; t < s.t1; ++t) {
        if (!q_ready) {
          if (!mbar_wait(smem_u32(&m.q_full), qcount & 1u, deadline, ab)) return false;
          q_ready = true;
        }
        const uint32_t slot = kcount % kIdxStages;
        if (!mbar_wait(smem_u32(&m.k_full[slot]), (kcount / kIdxStages) & 1u, deadline, ab)) return false;
        const uint32_t buf = acount & 1u;
        if (!mbar_wait(smem_u32(&m.acc_empty[buf]), ((acount >> 1) & 1u) ^ 1u, deadline, ab)) return false;
        tc_fence_after();
        const uint32_t d = tmem + buf * kIdxN;
        const uint32_t ka = sb + kIdxKOff + slot * kIdxKStage;
#pragma unroll
        for (int kk = 0; kk < kIdxD / 16; ++kk) {
          const uint32_t half = static_cast<uint32_t>(kk >> 2), off = static_cast<uint32_t>(kk & 3) * 32u;
          const uint64_t a = smem_desc(ka + half * kIdxKHalf + off, 16, 1024, SWZ_128B);
          const uint64_t b = smem_desc(sb + kIdxQOff + half * kIdxQHalf + off, 16, 1024, SWZ_128B);
          mma_bf16_ss(d, a, b, kIdesc, kk > 0 ? 1u : 0u);
        }
        mma_commit(smem_u32(&m.k_empty[slot]));
        mma_commit(smem_u32(&m.acc_full[buf]));
        ++kcount;
        ++acount;
      }
    }
    if (q_ready) {
      mma_commit(smem_u32(&m.q_empty));
      ++qcount;
    }
  }
  return true;
}

// Epilogue warp e (0..7): TMEM lane quarter = warp % 4, and the group's
// half e / 4 of its (row, head) columns (128 of the 256).  The columns are
// read 64 at a time with the 16x256b shape: thread t holds 16 of them (the
// same 16 on every tile, so their head weights stay in registers for the
// whole item) for 4 positions of the quarter, t/4 + {0, 8, 16, 24}.  A
// thread sums its 16 heads per position; a transpose-reduce over the 4
// threads that share the positions (lane bits 0..1) leaves each thread the
// full score of one position.
template <int H>
__device__ __forceinline__ bool idx_epilogue(const IdxParams& p, IdxMisc& m, const uint8_t* sbase, uint32_t tmem,
                                             const int32_t* cq, const int32_t* ck, int e) {
  constexpr int G = kIdxN / H;
  constexpr int GH = G / 2;          // rows per half
  constexpr int RB = 64 / H;         // rows per 64-column batch (H <= 64)
  constexpr int NB = GH / RB;        // batches per half: 2
  constexpr int JR = 8 / RB;         // 8-column repetitions per row
  static_assert(GH * H == 128 && NB == 2, "epilogue batching");
  const volatile int* ab = &m.abort_flag;
  const int lane = static_cast<int>(lane_id());
  const int quarter = static_cast<int>(threadIdx.x >> 5) & 3;
  const int half = e >> 2;
  const int li = lane & 3;
  const float* wsm = reinterpret_cast<const float*>(sbase + kIdxWOff);
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
  // the position this thread's final score belongs to, within the quarter
  const int my_pos = (lane >> 2) + 8 * li;
  uint32_t acount = 0, wcount = 0;
  const long long n_items = static_cast<long long>(p.groups) * p.kv_chunks;
  for (long long it = blockIdx.x; it < n_items; it += gridDim.x) {
    const uint64_t deadline = global_timer_ns() + p.timeout_ns;
    IdxWalk w;
    w.start(p, cq, it);
    IdxSeg s;
    bool first = true;
    float wr[NB][16];   // head weights of this thread's 16 columns per batch
    while (w.next(p, cq, ck, s)) {
      if (s.t1 <= s.t0) continue;
      if (first) {
        first = false;
        const uint32_t b = wcount & 1u;
        if (!mbar_wait(smem_u32(&m.w_full[b]), (wcount >> 1) & 1u, deadline, ab)) return false;
        const float* wb = wsm + b * kIdxN + half * 128;
#pragma unroll
        for (int bt = 0; bt < NB; ++bt)
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float2 x = *reinterpret_cast<const float2*>(wb + bt * 64 + 8 * j + 2 * li);
            wr[bt][2 * j] = x.x;
            wr[bt][2 * j + 1] = x.y;
          }
      }
      // this half's rows in the segment and the positions each sees
      int vis[GH];
      bool on[GH];
#pragma unroll
      for (int jj = 0; jj < GH; ++jj) {
        const int r = w.r_first + half * GH + jj;
        on[jj] = r >= s.r_begin && r < s.r_end;
        long long v = on[jj] ? idx_visible(cq, ck, s.b, r) : 0;
        if (v > p.row_stride) {
          if (lane == 0) atomicCAS(&g_device_error, 0, static_cast<int>(kErrIdxRowTooLong));
          v = p.row_stride;
        }
        on[jj] = on[jj] && v > p.skip_len;
        vis[jj] = static_cast<int>(v);
      }
      for (int t = s.t0; t < s.t1; ++t) {
        const uint32_t buf = acount & 1u;
        if (!mbar_wait(smem_u32(&m.acc_full[buf]), (acount >> 1) & 1u, deadline, ab)) return false;
        tc_fence_after();
        const int pos = t * kIdxTile + quarter * 32 + my_pos;
        // Paged cache: the quarter's 32 positions share one page; a page past
        // the table or outside the pool gives them no key, and score -inf.
        bool has_key = true;
        if (p.block_table != nullptr) {
          const int pg = t * (kIdxTile / kIdxPage) + quarter * 32 / kIdxPage;
          const int blk = pg < p.max_blocks ? __ldg(p.block_table + static_cast<size_t>(s.b) * p.max_blocks + pg) : -1;
          has_key = blk >= 0 && blk < p.num_blocks;
        }
#pragma unroll
        for (int bt = 0; bt < NB; ++bt) {
          bool any = false;
#pragma unroll
          for (int rr = 0; rr < RB; ++rr) any = any || on[bt * RB + rr];
          float xa[32], xb[32];   // positions +0/+8 and +16/+24 of the quarter
          if (any) {   // warp-uniform
            const uint32_t col = buf * kIdxN + static_cast<uint32_t>(half * 128 + bt * 64);
            tmem_ld16x256_x8(lane_base + col, xa);
            tmem_ld16x256_x8(lane_base + (16u << 16) + col, xb);
          }
          tmem_wait_ld();
          if (bt == NB - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&m.acc_empty[buf]));
          }
#pragma unroll
          for (int rr = 0; rr < RB; ++rr) {
            const int jj = bt * RB + rr;
            if (!on[jj]) continue;   // warp-uniform
            // partial sums of this thread's heads of row jj at its 4 positions
            float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f, c0 = 0.f, c1 = 0.f, d0 = 0.f, d1 = 0.f;
#pragma unroll
            for (int j = rr * JR; j < (rr + 1) * JR; ++j) {
              const float w0 = wr[bt][2 * j], w1 = wr[bt][2 * j + 1];
              ffma2(a0, a1, fmaxf(xa[4 * j + 0], 0.f), fmaxf(xa[4 * j + 1], 0.f), w0, w1);
              ffma2(b0, b1, fmaxf(xa[4 * j + 2], 0.f), fmaxf(xa[4 * j + 3], 0.f), w0, w1);
              ffma2(c0, c1, fmaxf(xb[4 * j + 0], 0.f), fmaxf(xb[4 * j + 1], 0.f), w0, w1);
              ffma2(d0, d1, fmaxf(xb[4 * j + 2], 0.f), fmaxf(xb[4 * j + 3], 0.f), w0, w1);
            }
            // positions +0, +8, +16, +24: transpose-reduce over lane bits 0..1
            const float v0 = a0 + a1, v1 = b0 + b1, v2 = c0 + c1, v3 = d0 + d1;
            float k0 = (li & 2) ? v2 : v0, k1 = (li & 2) ? v3 : v1;
            const float s0 = (li & 2) ? v0 : v2, s1 = (li & 2) ? v1 : v3;
            k0 += __shfl_xor_sync(0xffffffffu, s0, 2);
            k1 += __shfl_xor_sync(0xffffffffu, s1, 2);
            float sc = (li & 1) ? k1 : k0;
            sc += __shfl_xor_sync(0xffffffffu, (li & 1) ? k0 : k1, 1);
            if (pos < vis[jj]) {
              const int r = w.r_first + half * GH + jj;
              p.scores[static_cast<long long>(r - p.row0) * p.row_stride + pos] = has_key ? sc : -INFINITY;
            }
          }
        }
        ++acount;
      }
    }
    if (!first) {
      // every read of this item's weights is done
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&m.w_empty[wcount & 1u]));
      ++wcount;
    }
  }
  return true;
}

template <int H>
__global__ void __launch_bounds__(kIdxThreads, 1) dsa_scores_kernel(const __grid_constant__ IdxParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sbase = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  IdxMisc& m = *reinterpret_cast<IdxMisc*>(sbase + kIdxMiscOff);
  int32_t* cq = reinterpret_cast<int32_t*>(sbase + kIdxCuOff);
  int32_t* ck = cq + (kIdxMaxBatch + 1);
  const int warp = static_cast<int>(threadIdx.x >> 5);
  const int lane = static_cast<int>(lane_id());
  const uint32_t sb = smem_u32(sbase);

  if (p.block_table != nullptr) {
    // Paged cache: request b owns query rows [b s_next, (b + 1) s_next) and
    // seqlens[b] positions; ck holds their prefix sums, so that every
    // visibility rule reads lengths as for packed sequences.
    for (int i = static_cast<int>(threadIdx.x); i <= p.batch; i += kIdxThreads) cq[i] = i * p.s_next;
    if (warp == 0) {
      int base = 0;
      if (lane == 0) ck[0] = 0;
      for (int i0 = 0; i0 < p.batch; i0 += 32) {
        const int i = i0 + lane;
        int v = i < p.batch ? p.seqlens[i] : 0;
        v = v < 0 ? 0 : v;
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        if (i < p.batch) ck[i + 1] = base + incl;
        base += __shfl_sync(0xffffffffu, incl, 31);
      }
    }
  } else if (p.cu_q != nullptr) {
    for (int i = static_cast<int>(threadIdx.x); i <= p.batch; i += kIdxThreads) {
      cq[i] = p.cu_q[i];
      ck[i] = p.cu_kv[i];
    }
  } else if (threadIdx.x == 0) {
    cq[0] = 0;
    cq[1] = p.total_q;
    ck[0] = 0;
    ck[1] = p.total_kv;
  }
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&m.q_full), 1);
    mbar_init(smem_u32(&m.q_empty), 1);
    for (int i = 0; i < kIdxStages; ++i) {
      mbar_init(smem_u32(&m.k_full[i]), 1);
      mbar_init(smem_u32(&m.k_empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&m.acc_full[i]), 1);
      mbar_init(smem_u32(&m.acc_empty[i]), 8);   // one arrival per epilogue warp
      mbar_init(smem_u32(&m.w_full[i]), 1);
      mbar_init(smem_u32(&m.w_empty[i]), 8);
    }
    mbar_init(smem_u32(&m.drain), 1);
    m.abort_flag = 0;
    m.prior_error = *reinterpret_cast<volatile int*>(&g_device_error);
    fence_mbar_init();
    prefetch_tmap(&p.map_q);
    prefetch_tmap(&p.map_k);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&m.tmem_base), kIdxTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = m.tmem_base;

  if (m.prior_error == 0) {
    if (warp == 0) {
      if (lane == 0) {
        uint32_t kcount = 0, qcount = 0, wcount = 0;
        if (!idx_producer(p, m, sb, cq, ck, kcount, qcount, wcount)) idx_raise(m, kErrIdxProducerWait);
        // Drain: the copies this thread issued have landed before the CTA
        // exits, whether or not the consumers got to them (only the last
        // fill of each buffer can still be in flight).
        const int never = 0;
        const uint64_t dl = global_timer_ns() + 100000000ull;
        for (uint32_t i = kcount > kIdxStages ? kcount - kIdxStages : 0; i < kcount; ++i)
          mbar_wait(smem_u32(&m.k_full[i % kIdxStages]), (i / kIdxStages) & 1u, dl, &never);
        if (qcount > 0) mbar_wait(smem_u32(&m.q_full), (qcount - 1) & 1u, dl, &never);
        for (uint32_t i = wcount > 2 ? wcount - 2 : 0; i < wcount; ++i)
          mbar_wait(smem_u32(&m.w_full[i & 1u]), (i >> 1) & 1u, dl, &never);
      }
      __syncwarp();
    } else if (warp == 1) {
      if (lane == 0) {
        if (!idx_mma(p, m, sb, tmem, cq, ck)) idx_raise(m, kErrIdxMmaWait);
        // Drain: every MMA issued completes before TMEM is freed.
        const int never = 0;
        mma_commit(smem_u32(&m.drain));
        mbar_wait(smem_u32(&m.drain), 0, global_timer_ns() + 100000000ull, &never);
      }
      __syncwarp();
    } else {
      if (!idx_epilogue<H>(p, m, sbase, tmem, cq, ck, warp - kIdxEpiWarp0)) idx_raise(m, kErrIdxEpilogueWait);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kIdxTmemCols);
}

// ------------------------------------------------------------------ top-k

constexpr int kTopkMaxWarps = 32;   // CTAs of 256 threads, or 1024 for long rows
constexpr int kTopkBins = 2048;

struct TopkParams {
  const float* scores;        // [n_rows, row_stride]
  int32_t* indices;           // [total_q, topk]: rows row0 .. row0 + n_rows - 1 are written
  const int32_t* cu_q;        // [batch + 1], null for one dense sequence or a paged cache
  const int32_t* cu_kv;
  const int32_t* seqlens;     // paged cache: [batch] positions per request, else null
  const int32_t* block_table; // paged cache: [batch, max_blocks] (short rows list keyed positions only)
  int s_next;                 // paged cache: query rows per request
  int max_blocks, num_blocks; // paged cache
  long long row_stride;
  int total_q, total_kv, batch;
  int row0, n_rows, topk;
  int stage_cap;              // rows of at most this many positions are staged (a multiple of 4)
};

// Order-preserving image of an fp32 score: a < b as floats iff key(a) <
// key(b) as unsigned integers (NaN images sort by their bit pattern).
__device__ __forceinline__ uint32_t topk_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return u ^ ((u & 0x80000000u) ? 0xFFFFFFFFu : 0x80000000u);
}

// Image of -inf: keys at or below it (-inf, and NaNs with the sign bit set)
// are never selected.
constexpr uint32_t kKeyNegInf = 0x007FFFFFu;

// Shared state of one row's selection.
struct TopkShared {
  int scan[kTopkMaxWarps];
  int scan2[kTopkMaxWarps];
  int seq, krem, fin;
  uint32_t bin;
};

// The bin of `hist` (nbins bins, counts of the current class) that holds
// the class's krem-th largest key, and krem's rank inside it.  Thread t
// owns bins [t per, t per + per); the counts above come from a suffix scan.
// Ends with the block synchronised and sh.bin / sh.krem set.
template <int T>
__device__ __forceinline__ void topk_find_bin(const uint32_t* hist, int nbins, int krem, TopkShared& sh) {
  const int tid = static_cast<int>(threadIdx.x), lane = static_cast<int>(lane_id()), w = tid >> 5;
  const int per = nbins / T;
  int own = 0;
  for (int i = 0; i < per; ++i) own += static_cast<int>(hist[tid * per + i]);
  int incl = own;   // over this lane and the lanes above it
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_down_sync(0xffffffffu, incl, o);
    if (lane + o < 32) incl += y;
  }
  if (lane == 0) sh.scan[w] = incl;
  __syncthreads();
  int above = incl - own;
#pragma unroll
  for (int i = 0; i < (T / 32); ++i) above += i > w ? sh.scan[i] : 0;
  if (above < krem && krem <= above + own) {
    int acc = above;
    for (int i = per - 1; i >= 0; --i) {
      const int c = static_cast<int>(hist[tid * per + i]);
      if (krem <= acc + c) {
        sh.bin = static_cast<uint32_t>(tid * per + i);
        sh.krem = krem - acc;
        break;
      }
      acc += c;
    }
  }
  __syncthreads();
}

// Four consecutive keys starting at position 4 q (q < ceil(n / 4)); keys at
// or past n read as 0 and are masked by the callers.
template <bool kStaged>
__device__ __forceinline__ uint4 topk_keys4(const uint32_t* keys, const float* row, int q, int n) {
  if constexpr (kStaged) {
    return reinterpret_cast<const uint4*>(keys)[q];
  } else {
    uint4 k;
    const int s = 4 * q;
    k.x = s + 0 < n ? topk_key(row[s + 0]) : 0u;
    k.y = s + 1 < n ? topk_key(row[s + 1]) : 0u;
    k.z = s + 2 < n ? topk_key(row[s + 2]) : 0u;
    k.w = s + 3 < n ? topk_key(row[s + 3]) : 0u;
    return k;
  }
}

// Exclusive prefix over the block (in thread order) of two per-thread
// counts.  Ends with the block synchronised.
template <int T>
__device__ __forceinline__ void topk_block_scan2(int a, int b, TopkShared& sh, int& a_ex, int& b_ex) {
  const int lane = static_cast<int>(lane_id()), w = static_cast<int>(threadIdx.x >> 5);
  int ai = a, bi = b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(0xffffffffu, ai, o);
    const int y = __shfl_up_sync(0xffffffffu, bi, o);
    if (lane >= o) {
      ai += x;
      bi += y;
    }
  }
  if (lane == 31) {
    sh.scan[w] = ai;
    sh.scan2[w] = bi;
  }
  __syncthreads();
  int wa = 0, wb = 0;
#pragma unroll
  for (int i = 0; i < (T / 32); ++i) {
    wa += i < w ? sh.scan[i] : 0;
    wb += i < w ? sh.scan2[i] : 0;
  }
  a_ex = wa + ai - a;
  b_ex = wb + bi - b;
  __syncthreads();
}

// Selection of one row of n > topk positions (keys staged in shared memory
// or read from the row in global memory on every pass).
template <int T, bool kStaged>
__device__ __forceinline__ void topk_select(const float* row, int n, int topk, int32_t* out, uint32_t* hist,
                                            const uint32_t* keys, TopkShared& sh) {
  const int tid = static_cast<int>(threadIdx.x);
  const int nq = (n + 3) >> 2;
  if (tid == 0) sh.fin = 0;
  __syncthreads();
  // digits of 11, 11 and 10 bits; each pass counts the keys of the current
  // class (those sharing the digits fixed so far)
  uint32_t prefix = 0, pmask = 0;
  int krem = topk;
  for (int d = 0; d < 3; ++d) {
    const int shift = d == 0 ? 21 : (d == 1 ? 10 : 0);
    const uint32_t bmask = d == 2 ? 1023u : 2047u;
    if (d > 0) {
      for (int i = tid; i < kTopkBins; i += T) hist[i] = 0;
      __syncthreads();
    }
    int fin = 0;   // first pass: this thread's selectable keys (above -inf)
    for (int q = tid; q < nq; q += T) {
      const uint4 k = topk_keys4<kStaged>(keys, row, q, n);
      const int s = 4 * q;
      if ((k.x & pmask) == prefix) atomicAdd(&hist[(k.x >> shift) & bmask], 1u);
      if (s + 1 < n && (k.y & pmask) == prefix) atomicAdd(&hist[(k.y >> shift) & bmask], 1u);
      if (s + 2 < n && (k.z & pmask) == prefix) atomicAdd(&hist[(k.z >> shift) & bmask], 1u);
      if (s + 3 < n && (k.w & pmask) == prefix) atomicAdd(&hist[(k.w >> shift) & bmask], 1u);
      if (d == 0)
        fin += (k.x > kKeyNegInf) + (s + 1 < n && k.y > kKeyNegInf) + (s + 2 < n && k.z > kKeyNegInf) +
               (s + 3 < n && k.w > kKeyNegInf);
    }
    if (d == 0) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) fin += __shfl_xor_sync(0xffffffffu, fin, o);
      if ((tid & 31) == 0 && fin) atomicAdd(&sh.fin, fin);
    }
    __syncthreads();
    if (d == 0 && sh.fin <= topk) {
      // At most topk selectable keys: take every key above -inf (the
      // compaction below with the class "above -inf" and none of it partial).
      prefix = kKeyNegInf;
      pmask = 0xFFFFFFFFu;
      krem = 0;
      break;
    }
    topk_find_bin<T>(hist, static_cast<int>(bmask) + 1, krem, sh);
    prefix |= sh.bin << shift;
    pmask |= bmask << shift;
    krem = sh.krem;
    const bool whole = static_cast<int>(hist[sh.bin]) == krem;   // the class is taken whole
    __syncthreads();
    if (whole) break;
  }

  // Ordered compaction: keys above the class, then the first krem of the
  // class by position.  Thread t owns the quads [t QL, t QL + QL) with QL
  // odd (so the 16-byte reads of eight consecutive threads hit distinct
  // banks): it counts both kinds, one block scan gives the counts before
  // its run, and a second walk writes its picks in order.
  const int QL = ((nq + T - 1) / T) | 1;
  const int q0 = tid * QL < nq ? tid * QL : nq, q1 = q0 + QL < nq ? q0 + QL : nq;
  int gt = 0, eq = 0;
  for (int q = q0; q < q1; ++q) {
    const uint4 k = topk_keys4<kStaged>(keys, row, q, n);
    const int s = 4 * q;
    const uint32_t h0 = k.x & pmask, h1 = k.y & pmask, h2 = k.z & pmask, h3 = k.w & pmask;
    gt += (h0 > prefix) + (s + 1 < n && h1 > prefix) + (s + 2 < n && h2 > prefix) + (s + 3 < n && h3 > prefix);
    eq += (h0 == prefix) + (s + 1 < n && h1 == prefix) + (s + 2 < n && h2 == prefix) +
          (s + 3 < n && h3 == prefix);
  }
  int gt_ex, eq_ex;
  topk_block_scan2<T>(gt, eq, sh, gt_ex, eq_ex);
  int pos = gt_ex + (eq_ex < krem ? eq_ex : krem);
  int eq_seen = eq_ex;
  for (int q = q0; q < q1; ++q) {
    const uint4 k = topk_keys4<kStaged>(keys, row, q, n);
    const int s = 4 * q;
    const uint32_t kk[4] = {k.x, k.y, k.z, k.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t hi = kk[j] & pmask;
      bool take = s + j < n && hi > prefix;
      if (s + j < n && hi == prefix) {
        take = eq_seen < krem;
        ++eq_seen;
      }
      if (take) out[pos++] = s + j;
    }
  }
  // fewer selectable keys than topk: pad with -1
  const int picked = sh.fin < topk ? sh.fin : topk;
  for (int i = picked + tid; i < topk; i += T) out[i] = -1;
}

template <int T>
__global__ void __launch_bounds__(T, T == 256 ? 4 : 1) dsa_topk_kernel(const __grid_constant__ TopkParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem_raw);      // [kTopkBins]
  uint32_t* keys = hist + kTopkBins;                           // [stage_cap]
  __shared__ TopkShared sh;
  const int tid = static_cast<int>(threadIdx.x);
  const int r = p.row0 + static_cast<int>(blockIdx.x);

  // the row's sequence and visible length
  if (tid == 0) sh.seq = p.cu_q == nullptr ? 0 : -1;
  __syncthreads();
  if (p.cu_q != nullptr) {
    for (int i = tid; i < p.batch; i += T)
      if (p.cu_q[i] <= r && r < p.cu_q[i + 1]) sh.seq = i;
  }
  for (int i = tid; i < kTopkBins; i += T) hist[i] = 0;
  __syncthreads();
  const int b = sh.seq;
  long long v = 0;
  if (p.seqlens != nullptr) {   // paged cache: request r / s_next, its last s_next positions are the rows
    const int rb = r / p.s_next;
    const int lk = p.seqlens[rb];
    int cq2[2] = {rb * p.s_next, (rb + 1) * p.s_next}, ck2[2] = {0, lk < 0 ? 0 : lk};
    v = idx_visible(cq2, ck2, 0, r);
  } else if (b >= 0) {
    int cq2[2] = {0, p.total_q}, ck2[2] = {0, p.total_kv};
    if (p.cu_q != nullptr) {
      cq2[0] = p.cu_q[b];
      cq2[1] = p.cu_q[b + 1];
      ck2[0] = p.cu_kv[b];
      ck2[1] = p.cu_kv[b + 1];
    }
    v = idx_visible(cq2, ck2, 0, r);
  }
  int32_t* out = p.indices + static_cast<long long>(r) * p.topk;
  if (v > p.topk && p.scores == nullptr) {   // called for short rows only, but this one is longer
    if (tid == 0) atomicCAS(&g_device_error, 0, static_cast<int>(kErrIdxRowTooLong));
    v = p.topk;
  }
  if (v <= p.topk) {
    if (p.block_table == nullptr) {
      for (int i = tid; i < p.topk; i += T) out[i] = i < v ? i : -1;
      return;
    }
    // Paged cache: the positions that have a key, in order (a page past the
    // table or outside the pool has none), padded with -1.  Thread t owns a
    // run of pages; one block scan places its positions.
    const int32_t* btr = p.block_table + static_cast<long long>(r / p.s_next) * p.max_blocks;
    const int vv = static_cast<int>(v);
    const int npg = (vv + kIdxPage - 1) / kIdxPage;
    const int per = (npg + T - 1) / T;
    const int g0 = tid * per < npg ? tid * per : npg, g1 = g0 + per < npg ? g0 + per : npg;
    int cnt = 0;
    for (int g = g0; g < g1; ++g) {
      const int blk = g < p.max_blocks ? btr[g] : -1;
      if (blk >= 0 && blk < p.num_blocks) cnt += (vv - g * kIdxPage < kIdxPage ? vv - g * kIdxPage : kIdxPage);
    }
    int before, unused;
    topk_block_scan2<T>(cnt, 0, sh, before, unused);
    if (tid == T - 1) sh.krem = before + cnt;
    int o = before;
    for (int g = g0; g < g1; ++g) {
      const int blk = g < p.max_blocks ? btr[g] : -1;
      if (blk >= 0 && blk < p.num_blocks)
        for (int i = g * kIdxPage; i < vv && i < (g + 1) * kIdxPage; ++i) out[o++] = i;
    }
    __syncthreads();
    for (int i = sh.krem + tid; i < p.topk; i += T) out[i] = -1;
    return;
  }
  if (v > p.row_stride) {
    if (tid == 0) atomicCAS(&g_device_error, 0, static_cast<int>(kErrIdxRowTooLong));
    v = p.row_stride;
  }
  const int n = static_cast<int>(v);
  const float* row = p.scores + static_cast<long long>(blockIdx.x) * p.row_stride;
  if (n > p.stage_cap) {
    topk_select<T, false>(row, n, p.topk, out, hist, keys, sh);
    return;
  }
  // Stage the row's keys (16-byte loads, four in flight per thread, when the
  // row is 16-byte aligned); the tail of the last quad reads as 0.
  const int nq = (n + 3) >> 2;
  if ((reinterpret_cast<uintptr_t>(row) & 15u) == 0) {
    const float4* r4 = reinterpret_cast<const float4*>(row);
    uint4* k4 = reinterpret_cast<uint4*>(keys);
    const int full = n >> 2;
    for (int base = 0; base < full; base += 4 * T) {
      float4 t[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = base + u * T + tid;
        if (i < full) t[u] = __ldg(r4 + i);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = base + u * T + tid;
        if (i < full) k4[i] = make_uint4(topk_key(t[u].x), topk_key(t[u].y), topk_key(t[u].z), topk_key(t[u].w));
      }
    }
    for (int i = 4 * full + tid; i < 4 * nq; i += T) keys[i] = i < n ? topk_key(row[i]) : 0u;
  } else {
    for (int i = tid; i < 4 * nq; i += T) keys[i] = i < n ? topk_key(row[i]) : 0u;
  }
  __syncthreads();
  topk_select<T, true>(row, n, p.topk, out, hist, keys, sh);
}

}  // namespace smla
