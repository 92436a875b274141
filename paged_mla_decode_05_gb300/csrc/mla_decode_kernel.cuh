// Paged MLA decode kernel for sm_103a (GB300): the kernel template, included
// by the two translation units that instantiate it (mla_decode_sm103.cu: the
// paged mode; mla_decode_rows_sm103.cu: the row-list mode of the sparse
// decode), so the instances compile in parallel and neither carries the
// other's code.
//
// What it computes: for each work item (tokens [t0, t1) of request b) and each
// query head h, softmax(sm_scale * [q_nope|q_pe] . [c_kv|k_pe]^T) . c_kv over
// the item's tokens, gathered from the paged latent cache through the block
// table — the MLA decode of "SM100 Cutlass MLA decode with unrestricted
// num_heads (< 128) for DeepSeek TP" (vLLM PR #20769) and "[Kernel] Flashinfer
// MLA (trtllm-gen) decode kernel integration" (vLLM PR #21078). An item that
// covers a whole request writes out (bf16) and lse; a split item writes its
// normalised partial output and LSE for the combine kernel (the split-KV plus
// reduction scheme of PR #20769's bot summary).
//
// Design (GB300-first; the pages' kernels are prior art, not the blueprint):
// one 2-CTA cluster per work list, with split roles, because the fp32 output
// accumulator of 128 heads x 512 columns fills a whole SM's tensor memory:
//  * score CTA (cluster rank 0): streams 96-token KV tiles (all 576 columns)
//    into shared-memory stages, one TMA box per page piece (a page-aligned
//    run of 32 or 16 rows; per-SM TMA cost is per box, so few large boxes
//    keep up with HBM). The 4-D view lands every 8-row swizzle atom of the
//    tile at a fixed offset whichever page it came from, so one MMA spans the
//    whole tile. Q [128 heads x 576] stays in tensor memory (four loader
//    warps replace it between items); S = Q.K^T runs on tcgen05 (M = 128
//    heads, N = 96, A from tensor memory) from one issuer thread. The fp32
//    online softmax (one thread per head row, one pass per tile with a lazy
//    rescale) writes P and the per-row rescale record straight into the
//    output CTA's shared memory with asynchronous remote stores.
//  * output CTA (rank 1): holds O [128 x 512] fp32 in tensor memory, streams
//    V into a 3-slot ring with TMA (L2 hits: the score CTA just read the
//    same lines), issues O += P.V with tcgen05 (N = 256), applies the
//    rescale when the softmax maximum moved, and writes the normalised
//    output.
// FP8 (E4M3) cache, the template's second instance: K and V are read as
// bytes (576 per token, half the bf16 traffic) and multiplied on the tensor
// core in kind::f8f6f4. Q and P, which are not 8-bit quantities, enter the
// MMAs as two E4M3 terms each (hi + lo, about 8 significant bits, as bf16
// has), so each product is two MMAs; Q carries a per-row power-of-two scale
// and the per-tensor cache scale is applied in fp32 to the scores and the
// output.
// Heads below 128 are padded inside the kernel: zero Q rows in tensor memory
// and zero P rows in shared memory, never stored.
// Row-list mode (template flag ROWS, sparse decode): the tile's rows come
// from a per-request list of cache rows, copied by six warps of the pair
// with 16-byte cp.async into the same shared-memory layout (with the
// swizzle applied in the addresses); everything past the producers is the
// same code. TMA four-row gathers were measured first: at 512 bytes per
// instruction they ran at a third of this rate.
#pragma once

#include <cuda_runtime.h>

#include "mla_internal.h"
#include "ptx_sm103.cuh"

namespace mla {
namespace {

constexpr int kQPrefetchLead = 4;   // tiles before an item's end: L2 prefetch of the next Q

// Control block: identical offsets in both CTAs of the pair, so a barrier can
// be addressed in the peer by offset (mapa, multicast commit).
struct Ctrl {
  uint64_t kv_full[kF8NumStages];   // score: all pieces of a stage landed (TMA bytes)
  uint64_t kv_empty[kF8NumStages];  // score: S MMAs done reading the stage
  uint64_t s_full[2];             // score: S tile in tensor memory
  uint64_t s_free[2];             // score: softmax copied S out
  uint64_t q_ready[kNumPanels];   // score: Q of the next item in tensor memory, per panel
  uint64_t q_free;                // score: S MMAs of an item's last tile done (Q may be replaced)
  uint64_t p_empty[kNumPBufs];    // score: peer finished P.V on its P buffer k
  uint64_t v_full[kNumVSlots];    // output: V half landed
  uint64_t v_empty[kNumVSlots];   // output: P.V done reading the V half
  uint64_t p_full[kNumPBufs];     // output: P tile and row record landed (copy bytes)
  // output: the correction warps have taken tile g (and rescaled O if due).
  // 128 arrivals (the four correction warps, which run independently) per
  // phase, one phase per tile; a warp can be up to kNumPBufs - 1 tiles ahead
  // of another (it needs P of its tile, shipped after P.V of the tile
  // kNumPBufs earlier, which waited for every warp), so the ring has
  // kNumPBufs barriers and an early arrival never lands in a phase that a
  // slower warp has not completed.
  uint64_t o_ready[kNumPBufs];
  // output: P.V of tile g complete, ring of kNumPBufs. A waiter for tile t
  // always knows that P.V of tile t - kNumPBufs is complete (the correction
  // warps hold P of tile t + 1, or of t itself in the epilogue, which the
  // peer shipped after that P.V), and P.V of tile t + kNumPBufs cannot be
  // (it waits for them), so o_done[t % kNumPBufs] is in tile t's phase.
  uint64_t o_done[kNumPBufs];
  uint64_t o_drained[2];          // output: epilogue has read O columns [256h, 256h+256) of an item
  uint64_t qs_ready[kF8QScaleSlots];  // score (FP8): the Q row scales of an item are in their slot
  uint32_t tmem_base;
  int32_t p_seen;                 // output: P tiles received so far (paces the prefetcher)
};
static_assert(sizeof(Ctrl) <= kCtrlBytes, "control block too large");

constexpr uint32_t kIdescS = idesc_bf16_f32(128, kTile, 0, 0);   // K-major A and B
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 256, 0, 1);    // V is MN-major
constexpr uint32_t kIdescS8 = idesc_e4m3_f32(128, kTile, 0, 0);  // FP8: same shapes
constexpr uint32_t kIdescPV8 = idesc_e4m3_f32(128, 256, 0, 1);
constexpr uint32_t kFullMask = 0xffffffffu;
constexpr int kPrefetchTiles = 4;   // output prefetcher: distance ahead of received P (tiles)

// Lazy rescale threshold (log2 units): the running row maximum moves only
// when a tile's maximum exceeds it by more than this. bf16 P takes p up to
// 2^8. The FP8 path stores P as two E4M3 terms and scales it by
// 2^kF8PShift, so p * 2^kF8PShift <= 2^(threshold + shift) = 256 stays below
// E4M3's 448 while the smallest p kept (E4M3's 2^-9 subnormal step) is
// 2^-13 of the running maximum's weight.
template <bool F8> __host__ __device__ constexpr float rescale_threshold() { return F8 ? 4.0f : 8.0f; }
constexpr float kF8PShift = 4.0f;

template <bool F8> __host__ __device__ constexpr int num_stages() { return F8 ? kF8NumStages : kNumStages; }
template <bool F8> __host__ __device__ constexpr int stage_bytes() { return F8 ? kF8StageBytes : kStageBytes; }

MLA_DEVI int tiles_of(const WorkItem& it) {
  return it.t1 > it.t0 ? (it.t1 - it.t0 + kTile - 1) / kTile : 0;
}

// Work item i of the schedule. With lengths planned as upper bounds, its end
// is clamped to the request's length read from the device on every call, so
// one schedule (and one captured launch) serves any lengths up to the bounds.
MLA_DEVI WorkItem item_at(const DecodeParams& p, int i) {
  WorkItem w = p.items[i];
  w.len = w.seq_len;
  if (p.dynamic_lens) {
    w.len = max(0, min(w.seq_len, __ldg(&p.seq_lens[w.b])));
    w.t1 = max(w.t0, min(w.t1, w.len));
  }
  return w;
}

// End (exclusive) of the tokens that row `row` of item w attends to. With
// several query tokens per request (row = j * heads + h of the request),
// token j sees the request's first len - q_len + 1 + j tokens.
MLA_DEVI int row_end(const DecodeParams& p, const WorkItem& w, int row) {
  const int rr = w.h0 + row;
  if (p.q_len <= 1 || rr >= p.H) return w.t1;
  return min(w.t1, w.len - (p.q_len - 1) + rr / p.heads);
}

// Query heads of an item's head group: heads [h0, h0 + heads_of) of the
// request, at most 128 (the MMA M; fewer are padded inside the kernel).
MLA_DEVI int heads_of(const DecodeParams& p, const WorkItem& it) {
  return min(kMaxHeads, p.H - it.h0);
}

MLA_DEVI void report(const DecodeParams& p, uint32_t bits) {
  if (bits) atomicOr(p.err, bits);
}

// Optional timeline instrumentation (compiled only with -DMLA_TRACE): each
// role of the CTA pairs listed in the trace buffer records the SM clock at
// fixed points of every tile. Records time only; skips no work.
#ifdef MLA_TRACE
__device__ uint64_t* g_mla_trace = nullptr;   // [pairs][2 ranks][kTraceEvents][kTraceTiles]
constexpr int kTracePairs = 4, kTraceEvents = 64, kTraceTiles = 256;
// Slot 32 + ev records clock64 of event ev (SM cycles; comparable within one SM).
MLA_DEVI void trace(int ev, int g) {
  uint64_t* t = g_mla_trace;
  const int pair = static_cast<int>(cluster_id_x());
  if (t == nullptr || pair >= kTracePairs || g >= kTraceTiles) return;
  const int base = (pair * 2 + static_cast<int>(cluster_rank())) * kTraceEvents;
  t[(base + 32 + ev) * kTraceTiles + g] = static_cast<uint64_t>(clock64());
}
#define MLA_TRACE_AT(ev, g) trace(ev, g)
#else
#define MLA_TRACE_AT(ev, g) ((void)0)
#endif

// Block-table window of one producer warp: lane j holds the block id of page
// base + j of the current request, so one coalesced load serves 32 pages.
struct PageWindow {
  int base = -1;
  int val = 0;
};

// The pieces of one kTile-token tile: page-aligned runs of 32 rows (block
// size >= 32) or 16 rows (block size 16). A tile starts at a multiple of 96
// tokens, so at a multiple of 32, and every piece stays inside one page.
MLA_DEVI int pieces_per_tile(int block_size) {
  return block_size >= kRowsLargeBox ? kTile / kRowsLargeBox : kTile / kRowsSmallBox;
}
// Piece j of a tile: first row inside the tile and whether it is a 32-row box.
MLA_DEVI void piece_shape(int block_size, int j, int& r0, int& large) {
  large = block_size >= kRowsLargeBox;
  r0 = j * (large ? kRowsLargeBox : kRowsSmallBox);
}

// Make the warp's block-table window cover the pages of the tile starting at
// tile_t0 (all lanes call this together; lane i holds page base + i).
MLA_DEVI void window_cover(const DecodeParams& p, const WorkItem& w, int tile_t0,
                           PageWindow& win, int lane) {
  const int sh = __ffs(p.block_size) - 1;   // block sizes are powers of two
  const int first = tile_t0 >> sh;
  const int last = (min(tile_t0 + kTile, w.t1) - 1) >> sh;
  if (win.base < 0 || first < win.base || last >= win.base + 32) {
    win.base = first;
    const int n_pages = (w.t1 + p.block_size - 1) >> sh;
    win.val = (first + lane < n_pages)
                  ? __ldg(&p.block_table[static_cast<int64_t>(w.b) * p.max_blocks + first + lane])
                  : -1;
  }
}

// Cache row of token t through the window (all lanes call this together,
// each for its own t), or the first row past the pool (a TMA box there reads
// zeros) for tokens at or past the item's end and for out-of-range block ids
// (MLA_DEVERR_BAD_BLOCK).
MLA_DEVI int cache_row(const DecodeParams& p, const WorkItem& w, int t, const PageWindow& win,
                       uint32_t& err) {
  const int sh = __ffs(p.block_size) - 1;
  const int blk = __shfl_sync(kFullMask, win.val, ((t >> sh) - win.base) & 31);
  const int oob = static_cast<int>(p.num_blocks * p.block_size);
  if (t >= w.t1) return oob;
  if (blk < 0 || static_cast<int64_t>(blk) >= p.num_blocks) {
    err |= 1u;  // MLA_DEVERR_BAD_BLOCK
    return oob;
  }
  return (blk << sh) + (t & (p.block_size - 1));
}

// Lane 0 waits on a barrier; the whole warp learns the outcome.
MLA_DEVI bool warp_wait(uint32_t bar, uint32_t parity, int lane) {
  bool ok = true;
  if (lane == 0) ok = mbar_wait(bar, parity);
  return __shfl_sync(kFullMask, ok ? 1 : 0, 0) != 0;
}

// ------------------------------------------------------- row-list producers

// Warps that fetch the rows of a tile in row-list mode: the score CTA's
// producer and its two idle warps; the output CTA's producer and its five
// idle warps. Each full barrier counts one arrival per lane of them.
constexpr int kRowsScoreWarps = 3;
constexpr int kRowsOutWarps = 6;

// Cache rows of list positions tile_t0 + 32 j + lane (j < 3) of item w:
// positions at or past the item's end take the item's last row (the softmax
// masks them; any finite row serves), and a row outside the cache (not
// written by the row-list kernel) is replaced by row 0.
MLA_DEVI void tile_rows(const DecodeParams& p, const WorkItem& w, int tile_t0, int lane,
                        int (&rr)[3]) {
  const int n_rows = static_cast<int>(p.num_blocks * p.block_size);
  const int32_t* rl = p.rows + static_cast<int64_t>(w.b) * p.rows_stride;
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    const int t = min(tile_t0 + 32 * j + lane, w.t1 - 1);
    const int r = __ldg(&rl[t]);
    rr[j] = (r >= 0 && r < n_rows) ? r : 0;
  }
}
// Row of tile position pos (all lanes call this with positions in one
// 32-position block).
MLA_DEVI int row_at(const int (&rr)[3], int pos) {
  const int j = pos >> 5;
  const int v = j == 0 ? rr[0] : (j == 1 ? rr[1] : rr[2]);
  return __shfl_sync(kFullMask, v, pos & 31);
}

// Row-list producer, one of `parts` warps: each tile's rows are copied from
// the cache with 16-byte cp.async into the layout the paged mode's TMA boxes
// produce ([8-row group][128-byte panel][8 rows][128 B], the 128-byte
// swizzle XORing the 16-byte chunk index with the row's index in its group;
// FP8 rope columns: [group][8 rows][64 B], the 64-byte swizzle XORing with
// half the row index). Per warp instruction: 4 rows x 128 bytes, lanes
// 8q..8q+7 on row q. Warp `part` takes the row quads part, part + parts, ...
// Every lane arrives on the full barrier once its copies have landed
// (cp.async.mbarrier.arrive.noinc); the MMA issuer fences the generic-proxy
// writes before its tensor-core reads.
// OUT = false: the score CTA's K tiles (576 columns, ring of stages);
// OUT = true: the output CTA's V (512 columns; bf16 as two 256-column
// slots per tile, FP8 as one).
template <bool F8, bool OUT>
MLA_DEVI void rows_producer(const DecodeParams& p, Ctrl* c, uint8_t* data, int lane, int part,
                            int parts, int it0, int it1) {
  constexpr int NS = OUT ? kNumVSlots : num_stages<F8>();
  constexpr int SB = OUT ? kVHalfBytes : stage_bytes<F8>();
  constexpr int kSlotsPerTile = (OUT && !F8) ? 2 : 1;
  constexpr int kRowBytes = F8 ? kD : kD * 2;
  constexpr int kPanels = OUT ? (F8 ? kF8Panels : kVHalfPanels) : (F8 ? kF8Panels : kNumPanels);
  constexpr int kGroupBytes = F8 ? kF8NopeGroupBytes : (OUT ? kVGroupBytes : kKGroupBytes);
  const char* cache = static_cast<const char*>(p.kv_cache);
  const int q = lane >> 3, ch = lane & 7;
  uint32_t err = 0;
  int h = 0;
  bool ok = true;
  for (int it = it0; it < it1 && ok; ++it) {
    const WorkItem w = item_at(p, it);
    if (!OUT && part == 0 && lane == 0) {   // MLA_DEVERR_SEQLEN_MISMATCH: above the bound
      const int len = __ldg(&p.seq_lens[w.b]);
      if (len < 0 || len > w.seq_len) err |= 2u;
    }
    const int nt = tiles_of(w);
    for (int i = 0; i < nt && ok; ++i) {
      const int tile_t0 = w.t0 + i * kTile;
      int rr[3];
      tile_rows(p, w, tile_t0, lane, rr);
      for (int half = 0; half < kSlotsPerTile; ++half, ++h) {
        const int s = h % NS;
        const uint32_t empty = smem_addr(OUT ? &c->v_empty[s] : &c->kv_empty[s]);
        if (h >= NS && !warp_wait(empty, ((h / NS) - 1) & 1, lane)) {
          ok = false;
          break;
        }
        const uint32_t st = smem_addr(data + s * SB);
        const int col0 = (OUT && !F8) ? half * kVHalfPanels * 128 : 0;   // byte column
        for (int g4 = part; g4 < kTile / 4; g4 += parts) {
          const int pos = 4 * g4 + q;
          const int r8 = pos & 7;
          const char* src = cache + static_cast<int64_t>(row_at(rr, pos)) * kRowBytes + col0 + ch * 16;
          const uint32_t dst = st + (pos >> 3) * kGroupBytes + r8 * 128 + ((ch ^ r8) << 4);
#pragma unroll
          for (int k = 0; k < kPanels; ++k) cp_async16(dst + k * kAtomBytes, src + k * 128);
        }
        if (F8 && !OUT) {   // rope columns: 8 rows x 4 chunks per instruction
          const int c4 = lane & 3;
          for (int i8 = part; i8 < kTile / 8; i8 += parts) {
            const int pos = 8 * i8 + (lane >> 2);
            const int r8 = pos & 7;
            cp_async16(st + kF8NopeBytes + (pos >> 3) * kF8RopeGroupBytes + r8 * 64 +
                           ((c4 ^ (r8 >> 1)) << 4),
                       cache + static_cast<int64_t>(row_at(rr, pos)) * kRowBytes + kDc + c4 * 16);
          }
        }
        cp_async_arrive_noinc(smem_addr(OUT ? &c->v_full[s] : &c->kv_full[s]));
      }
    }
  }
  cp_async_wait_all();   // nothing of this warp is in flight when it leaves
  if (!ok) err |= 4u;
  err = __reduce_or_sync(kFullMask, err);
  if (lane == 0) report(p, err);
}

// ------------------------------------------------------------ score CTA roles

// TMA producer warp: each 96-token tile into stage g % stages, one 4-D box
// per page piece, lane j loading piece j. bf16: one box of all 9 panels. FP8:
// lanes 0..15 load the 512 c_kv columns (4 panels) and lanes 16..31 the 64
// rope columns of the same pieces. The stage layout does not depend on how
// the tile is cut into pieces; one barrier per stage counts the bytes of all
// pieces.
template <bool F8>
MLA_DEVI void score_producer(const DecodeParams& p, Ctrl* c, uint8_t* data, int lane, int it0,
                             int it1) {
  constexpr int NS = num_stages<F8>();
  constexpr int SB = stage_bytes<F8>();
  uint32_t err = 0;
  const uint64_t policy = policy_evict_normal();
  int g = 0;
  bool ok = true;
  const int n = pieces_per_tile(p.block_size);
  const int j = F8 ? (lane & 15) : lane;   // this lane's piece
  for (int it = it0; it < it1 && ok; ++it) {
    const WorkItem w = item_at(p, it);
    if (lane == 0) {   // MLA_DEVERR_SEQLEN_MISMATCH: not the planned length, or above the bound
      const int len = __ldg(&p.seq_lens[w.b]);
      if (p.dynamic_lens ? (len < 0 || len > w.seq_len) : len != w.seq_len) err |= 2u;
    }
    PageWindow win;
    const int nt = tiles_of(w);
    for (int i = 0; i < nt && ok; ++i, ++g) {
      // Warm L2 with the Q rows of the next non-empty item a few tiles before
      // they are loaded (earlier, the streaming cache would evict them).
      if (lane == 0 && i == max(nt - kQPrefetchLead, 0)) {
        for (int nx = it + 1; nx < it1; ++nx) {
          const WorkItem wn = item_at(p, nx);
          if (tiles_of(wn) == 0) continue;
          const int64_t qrow = static_cast<int64_t>(wn.b) * p.H + wn.h0;
          const int nh = heads_of(p, wn);
          const uint16_t* qn = p.q_nope + qrow * kDc;
          const uint16_t* qp = p.q_pe + qrow * kDr;
          asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(qn), "r"(nh * kDc * 2) : "memory");
          asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(qp), "r"(nh * kDr * 2) : "memory");
          break;
        }
      }
      const int s = g % NS;
      const int tile_t0 = w.t0 + i * kTile;
      int r0, large;
      piece_shape(p.block_size, j < n ? j : 0, r0, large);
      window_cover(p, w, tile_t0, win, lane);
      const int y = cache_row(p, w, tile_t0 + r0, win, err);   // a multiple of 8
      MLA_TRACE_AT(0, g);
      if (g >= NS && !warp_wait(smem_addr(&c->kv_empty[s]), ((g / NS) - 1) & 1, lane)) {
        ok = false;
        break;
      }
      const uint32_t full = smem_addr(&c->kv_full[s]);
      if (lane == 0) mbar_arrive_expect_tx(full, SB);
      __syncwarp();
      uint8_t* stage = data + s * SB;
      if (!F8) {
        if (lane < n)
          tma_load_4d(smem_addr(stage + (r0 >> 3) * kKGroupBytes),
                      large ? static_cast<const void*>(&p.tmap_k32)
                            : static_cast<const void*>(&p.tmap_k16),
                      0, 0, 0, y >> 3, full, policy);
      } else if (j < n) {
        if (lane < 16)
          tma_load_4d(smem_addr(stage + (r0 >> 3) * kF8NopeGroupBytes),
                      large ? static_cast<const void*>(&p.tmap_k32)
                            : static_cast<const void*>(&p.tmap_k16),
                      0, 0, 0, y >> 3, full, policy);
        else
          tma_load_3d(smem_addr(stage + kF8NopeBytes + (r0 >> 3) * kF8RopeGroupBytes),
                      large ? static_cast<const void*>(&p.tmap_v32)
                            : static_cast<const void*>(&p.tmap_v16),
                      0, 0, y >> 3, full, policy);
      }
      if (lane == 0) MLA_TRACE_AT(26, g);
    }
  }
  if (!ok) err |= 4u;
  err = __reduce_or_sync(kFullMask, err);
  if (lane == 0) report(p, err);
}

// S MMA issuer: S[g%2] = Q . K^T over the 576 columns with N = 96 (the
// whole tile: its 8-row atoms sit at fixed offsets in the stage whichever
// pages they came from). bf16: 36 k-steps of 16 columns. FP8: 18 k-steps of
// 32 columns, each issued twice, for the hi and the lo terms of Q (both in
// tensor memory) against the same K columns. An item's first tile follows
// its Q into tensor memory panel by panel; later tiles issue the fully
// unrolled sequence (one thread issues one MMA every ~45 cycles at best).
template <bool F8, bool ROWS>
MLA_DEVI void score_mma(const DecodeParams& p, Ctrl* c, uint8_t* data, uint32_t tmem, int it0,
                        int it1) {
  constexpr int NS = num_stages<F8>();
  constexpr int SB = stage_bytes<F8>();
  int g = 0, n_items = 0;
  bool ok = true;
  for (int it = it0; it < it1 && ok; ++it) {
    const WorkItem w = item_at(p, it);
    const int nt = tiles_of(w);
    if (nt == 0) continue;
    const uint32_t q_par = n_items & 1;
    ++n_items;
    for (int i = 0; i < nt; ++i, ++g) {
      const int s = g % NS;    // KV stage
      const int sb = g & 1;    // S buffer
      if (g >= 2 && !mbar_wait(smem_addr(&c->s_free[sb]), ((g >> 1) - 1) & 1)) { ok = false; break; }
      MLA_TRACE_AT(2, g);
      if (!mbar_wait(smem_addr(&c->kv_full[s]), (g / NS) & 1)) { ok = false; break; }
      MLA_TRACE_AT(1, g);
      tc_after_sync();
      if constexpr (ROWS) fence_proxy_async_smem();   // cp.async (generic proxy) data
      const uint32_t d = tmem + kTmemS0 + sb * kTile;
      const uint32_t a = tmem + kTmemQ;
      uint8_t* stage = data + s * SB;
      if (!F8) {
        // Descriptor of panel 0 (8-row atoms kKGroupBytes apart); later
        // k-steps only move the start-address field (low word, 16-byte units,
        // never carries out): +1 KB per panel, +32 B per k-step.
        const uint64_t bp = smem_desc(smem_addr(stage), 16, kKGroupBytes);
        const uint32_t hi = static_cast<uint32_t>(bp >> 32);
        const uint32_t blo = static_cast<uint32_t>(bp);
        if (i == 0) {
#pragma unroll 1
          for (int pc = 0; pc < kNumPanels; ++pc) {
            if (!mbar_wait(smem_addr(&c->q_ready[pc]), q_par)) { ok = false; break; }
            tc_after_sync();
#pragma unroll
            for (int q = 0; q < 4; ++q)
              mma_ts(d, a + pc * 32 + q * 8,
                     (static_cast<uint64_t>(hi) << 32) | (blo + pc * (kAtomBytes / 16) + q * 2),
                     kIdescS, (pc > 0 || q > 0) ? 1u : 0u);
          }
          if (!ok) break;
        } else {
#pragma unroll
          for (int kq = 0; kq < kNumPanels * 4; ++kq)   // panel kq/4, 32 bytes per k-step
            mma_ts(d, a + kq * 8,
                   (static_cast<uint64_t>(hi) << 32) | (blo + (kq >> 2) * (kAtomBytes / 16) + (kq & 3) * 2),
                   kIdescS, kq > 0 ? 1u : 0u);
        }
      } else {
        // c_kv columns: 128-byte panels 1 KB apart, 8-row groups
        // kF8NopeGroupBytes apart, 32 bytes per k-step; rope columns: one
        // 64-byte-swizzled panel, 8-row groups kF8RopeGroupBytes apart.
        const uint64_t kn = smem_desc(smem_addr(stage), 16, kF8NopeGroupBytes);
        const uint64_t kr = smem_desc(smem_addr(stage + kF8NopeBytes), 16, kF8RopeGroupBytes,
                                      kLayoutSw64);
        auto kdesc = [&](int ks) -> uint64_t {
          return ks < 16 ? kn + static_cast<uint64_t>((ks >> 2) * (kAtomBytes / 16) + (ks & 3) * 2)
                         : kr + static_cast<uint64_t>((ks - 16) * 2);
        };
        if (i == 0) {
          // Q arrives two k-steps (64 columns, hi and lo) per barrier.
#pragma unroll 1
          for (int pc = 0; pc < kNumPanels; ++pc) {
            if (!mbar_wait(smem_addr(&c->q_ready[pc]), q_par)) { ok = false; break; }
            tc_after_sync();
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              const int ks = 2 * pc + q;
              mma_ts_f8(d, a + ks * 8, kdesc(ks), kIdescS8, ks > 0 ? 1u : 0u);
              mma_ts_f8(d, a + kF8QLoCol + ks * 8, kdesc(ks), kIdescS8, 1u);
            }
          }
          if (!ok) break;
        } else {
#pragma unroll
          for (int ks = 0; ks < kD / 32; ++ks) {
            mma_ts_f8(d, a + ks * 8, kdesc(ks), kIdescS8, ks > 0 ? 1u : 0u);
            mma_ts_f8(d, a + kF8QLoCol + ks * 8, kdesc(ks), kIdescS8, 1u);
          }
        }
      }
      MLA_TRACE_AT(24, g);
      tc_commit(smem_addr(&c->kv_empty[s]));
      tc_commit(smem_addr(&c->s_full[sb]));
      if (i == nt - 1) tc_commit(smem_addr(&c->q_free));   // Q may now be replaced
      MLA_TRACE_AT(3, g);
    }
  }
  if (!ok) report(p, 4u);
}

// Load the Q rows of item w (request w.b, heads w.h0 ...) into tensor memory
// columns [0, 288): lane = head of the group, two bf16 per column. Lanes past
// the group's heads are zero (in-kernel head padding).
// The first three panels are loaded into registers first; then, when
// wait_parity >= 0, the warp waits for that phase of q_free (the S MMAs of
// the previous item's last tile are done) before it overwrites Q. Returns
// false if that wait ran out of time.
__device__ __noinline__ bool load_q(const DecodeParams& p, Ctrl* c, const WorkItem& w, int row,
                                    uint32_t trow, int wait_parity) {
  // The warp writes its 32-lane quarter of Q as two 16-lane halves in the
  // 16x256b fragment: a quad of threads reads 32 consecutive bytes of one head
  // row, so each load instruction fills whole sectors of 8 rows.
  const int lane = row & 31;
  const int q0 = row - lane;                    // first head of this quarter
  const int g4 = lane >> 2, u = lane & 3;
  const int64_t r0 = static_cast<int64_t>(w.b) * p.H + w.h0 + q0 + g4;
  const uint2* qn = reinterpret_cast<const uint2*>(p.q_nope + r0 * kDc) + u;
  const uint2* qp = reinterpret_cast<const uint2*>(p.q_pe + r0 * kDr) + u;
  const int nv = heads_of(p, w) - (q0 + g4);    // heads q0+g4+8m exist while 8m < nv
  // Panels stream through a ring of three register buffers: panel cc + 3 is
  // requested as soon as panel cc is in tensor memory, so three panels are in
  // flight throughout. Each panel is announced on its own barrier (one arrival
  // per warp), and the item's first S MMAs follow it panel by panel.
  uint2 v[3][4][4];   // [ring slot][head q0+g4+8m][32-byte column block]
  auto request = [&](int cc, uint2 (&dst)[4][4]) {
#pragma unroll
    for (int m = 0; m < 4; ++m)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        dst[m][e] = 8 * m < nv ? __ldg(cc < 8 ? qn + m * 8 * (kDc / 4) + cc * 16 + e * 4
                                              : qp + m * 8 * (kDr / 4) + e * 4)
                               : make_uint2(0u, 0u);
  };
#pragma unroll
  for (int cc = 0; cc < 3; ++cc) request(cc, v[cc]);
  if (wait_parity >= 0) {
    if (!__all_sync(kFullMask, mbar_wait(smem_addr(&c->q_free), static_cast<uint32_t>(wait_parity))))
      return false;
    tc_after_sync();
  }
#pragma unroll
  for (int cc = 0; cc < kNumPanels; ++cc) {
    uint2 (&cur)[4][4] = v[cc % 3];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t r[16];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        r[4 * e + 0] = cur[2 * h][e].x;
        r[4 * e + 1] = cur[2 * h][e].y;
        r[4 * e + 2] = cur[2 * h + 1][e].x;
        r[4 * e + 3] = cur[2 * h + 1][e].y;
      }
      tmem_st16x256b_x4(trow + (static_cast<uint32_t>(16 * h) << 16) + kTmemQ + cc * 32, r);
    }
    tmem_wait_st();
    tc_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&c->q_ready[cc]));
    if (cc + 3 < kNumPanels) request(cc + 3, cur);
  }
  return true;
}

// Panels [pc0, pc1) of the FP8 path's Q of item w, row `row` (64 columns
// each: two steps of 32 columns), scaled by inv_s = 2^-k and split into hi
// and lo E4M3 codes, into tensor memory; each panel is announced on its
// q_ready barrier. Called by the Q loader warps for panels 0..4 and by the
// softmax warps, idle until the item's first S tile, for panels 5..8: both
// halves of the conversion run at once at every item boundary.
constexpr int kQPanelsByLoader = 5;
__device__ __noinline__ bool convert_q_f8(const DecodeParams& p, Ctrl* c, const WorkItem& w,
                                          int row, uint32_t trow, float inv_s, int pc0, int pc1) {
  const int lane = row & 31;
  const bool active = row < heads_of(p, w);
  const int64_t r = static_cast<int64_t>(w.b) * p.H + w.h0 + (active ? row : 0);
  const uint4* qn = reinterpret_cast<const uint4*>(p.q_nope + r * kDc);   // 64 x 16 B
  const uint4* qp = reinterpret_cast<const uint4*>(p.q_pe + r * kDr);     // 8 x 16 B
  auto chunk = [&](int j) -> uint4 {   // 16-byte piece j < 72 of the row
    return active ? __ldg(j < kDc / 8 ? qn + j : qp + (j - kDc / 8)) : make_uint4(0u, 0u, 0u, 0u);
  };
  const uint64_t is2 = pack_f32x2(inv_s, inv_s);
  uint4 nxt[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) nxt[e] = chunk(8 * pc0 + e);
  // One 64-column panel (two steps of 32 columns, both terms) per pass, each
  // step in its own registers, so that one wait for the tensor-memory stores
  // per panel (before the panel is announced) covers both steps.
#pragma unroll 1
  for (int pc = pc0; pc < pc1; ++pc) {
    uint32_t hw[2][8], lw[2][8];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int cc = 2 * pc + h;
      uint4 v[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) v[e] = nxt[e];
      if (cc + 1 < 2 * pc1) {
#pragma unroll
        for (int e = 0; e < 4; ++e) nxt[e] = chunk(4 * (cc + 1) + e);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t wd[4] = {v[e].x, v[e].y, v[e].z, v[e].w};
#pragma unroll
        for (int k = 0; k < 4; k += 2) {
          // bf16 pairs (2 elements per word) -> fp32, scaled by 2^-k (exact).
          const uint32_t a = split_e4m3x2(mul_f32x2(pack_b32x2(wd[k] << 16, wd[k] & 0xFFFF0000u), is2));
          const uint32_t b =
              split_e4m3x2(mul_f32x2(pack_b32x2(wd[k + 1] << 16, wd[k + 1] & 0xFFFF0000u), is2));
          hw[h][2 * e + k / 2] = (a & 0xFFFFu) | (b << 16);
          lw[h][2 * e + k / 2] = (a >> 16) | (b & 0xFFFF0000u);
        }
      }
      tmem_st8(trow + kTmemQ + cc * 8, hw[h]);
      tmem_st8(trow + kTmemQ + kF8QLoCol + cc * 8, lw[h]);
    }
    // tcgen05.st reads its source registers asynchronously: complete the
    // stores before the registers are reused and before the panel is announced.
    tmem_wait_st();
    tc_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&c->q_ready[pc]));
  }
  return true;
}

// FP8 path: Q of item w as two E4M3 terms per element in tensor memory, hi
// codes in columns [0, 144) and lo codes in [144, 288) of lane `row`, with a
// per-row power-of-two scale: q = 2^k (hi + lo), where 2^k puts max|q| of
// the row in [128, 256). A bf16 q has 8 significant bits, so hi + lo holds it
// exactly unless |q| < 2^-9 max|q| (then the error is below 2^-17 max|q|).
// Each thread handles its own row: a first pass over the row finds max|q|
// (as the largest bf16 magnitude pattern, whose order is that of the
// values), writes 2^k into qscale (the ring slot of this item) and arrives on
// qs_ready[slot]; then, when wait_parity >= 0, the warp waits on q_free and
// converts panels 0..4 of the row (convert_q_f8; the softmax warps convert
// panels 5..8 at the same time). Rows past the group's heads are zero.
__device__ __noinline__ bool load_q_f8(const DecodeParams& p, Ctrl* c, float* qscale,
                                       const WorkItem& w, int row, uint32_t trow,
                                       int wait_parity, int slot) {
  const int lane = row & 31;
  const bool active = row < heads_of(p, w);
  const int64_t r = static_cast<int64_t>(w.b) * p.H + w.h0 + (active ? row : 0);
  const uint4* qn = reinterpret_cast<const uint4*>(p.q_nope + r * kDc);   // 64 x 16 B
  const uint4* qp = reinterpret_cast<const uint4*>(p.q_pe + r * kDr);     // 8 x 16 B
  auto chunk = [&](int j) -> uint4 {   // 16-byte piece j < 72 of the row
    return active ? __ldg(j < kDc / 8 ? qn + j : qp + (j - kDc / 8)) : make_uint4(0u, 0u, 0u, 0u);
  };
  uint32_t mx = 0;
#pragma unroll 8
  for (int j = 0; j < kD / 8; ++j) {
    const uint4 v = chunk(j);
    mx = __vmaxu2(mx, __vmaxu2(__vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu),
                               __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu)));
  }
  mx = max(mx & 0xFFFFu, mx >> 16);
  // Biased exponent E of max|q| (clamped so 2^k and 2^-k are normal fp32):
  // max|q| / 2^k lies in [128, 256) for k = E - 134.
  const int E = min(254, max(8, static_cast<int>(mx >> 7)));
  const float inv_s = __uint_as_float(static_cast<uint32_t>(261 - E) << 23);   // 2^-k
  qscale[slot * kMaxHeads + row] = __uint_as_float(static_cast<uint32_t>(E - 7) << 23);   // 2^k
  mbar_arrive(smem_addr(&c->qs_ready[slot]));
  if (wait_parity >= 0) {
    if (!__all_sync(kFullMask, mbar_wait(smem_addr(&c->q_free), static_cast<uint32_t>(wait_parity))))
      return false;
    tc_after_sync();
  }
  return convert_q_f8(p, c, w, row, trow, inv_s, 0, kQPanelsByLoader);
}

// Q loader warps (one per tensor-memory lane quadrant): the Q of each of the
// pair's items in turn, so the softmax warps never stop for it. Each call
// reads the next item's Q right after the previous Q is written (bf16: its
// first panels into registers; FP8: the row maxima and scales), then waits
// on q_free for the S MMAs of the previous item's last tile (phase j - 1 for
// the j-th non-empty item: the barrier cannot run ahead, since item j's last
// tile needs this Q first).
template <bool F8>
MLA_DEVI void score_qloader(const DecodeParams& p, Ctrl* c, uint8_t* data, uint32_t tmem,
                            int warp, int lane, int it0, int it1) {
  const int row = (warp & 3) * 32 + lane;
  const uint32_t trow = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
  float* qscale = reinterpret_cast<float*>(data + kF8NumStages * kF8StageBytes);
  int n_items = 0;
  for (int it = it0; it < it1; ++it) {
    if (tiles_of(item_at(p, it)) == 0) continue;
    const int wait_parity = n_items > 0 ? (n_items - 1) & 1 : -1;
    const bool ok = F8 ? load_q_f8(p, c, qscale, item_at(p, it), row, trow, wait_parity,
                                   n_items % kF8QScaleSlots)
                       : load_q(p, c, item_at(p, it), row, trow, wait_parity);
    if (!ok) {
      if (lane == 0) report(p, 4u);
      return;
    }
    ++n_items;
  }
}

// One pass of the softmax over a tile's 96 raw scores r (columns at or past
// the item's end already set to -inf): p = 2^(s*scale*log2e - m) rounded to
// bf16, written in 12 core-matrix chunks of 8 tokens straight into the output
// CTA's P buffer (p_dst, 128 B apart) with remote stores counted on its
// p_full barrier; returns the row sum of the p values (fp32, before rounding).
MLA_DEVI float softmax_tile(const uint32_t (&r)[kTile], uint64_t sl2x2, uint64_t negm2,
                            uint32_t p_dst, uint32_t peer_bar) {
  uint64_t ls2 = pack_f32x2(0.0f, 0.0f);
#pragma unroll
  for (int q = 0; q < kTile / 8; ++q) {
    uint32_t pk[4];
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
      float d0, d1;
      unpack_f32x2(fma_f32x2(pack_b32x2(r[8 * q + j], r[8 * q + j + 1]), sl2x2, negm2), d0, d1);
      const float e0 = fast_exp2(d0);
      const float e1 = fast_exp2(d1);
      ls2 = add_f32x2(ls2, pack_f32x2(e0, e1));
      pk[j / 2] = pack_bf16x2(e0, e1);
    }
    st_async_v4(p_dst + q * 128, pk[0], pk[1], pk[2], pk[3], peer_bar);
  }
  float ls0, ls1;
  unpack_f32x2(ls2, ls0, ls1);
  return ls0 + ls1;
}

// FP8 path: the same pass with p' = 2^(s * c - m') stored as two E4M3 terms
// (split_e4m3x2): 16-token chunks of hi codes into core-matrix columns 0..5
// of the row and the matching lo codes into columns 6..11. The p' values of
// a chunk replace its scores in r (the role's register budget has no room
// for a second copy). Returns the row sum of the p' values (fp32, before the
// split).
MLA_DEVI float softmax_tile_f8(uint32_t (&r)[kTile], uint64_t c2, uint64_t negm2,
                               uint32_t p_dst, uint32_t peer_bar) {
  uint64_t ls2 = pack_f32x2(0.0f, 0.0f);
#pragma unroll
  for (int q = 0; q < kTile / 16; ++q) {
#pragma unroll
    for (int j = 16 * q; j < 16 * q + 16; j += 2) {
      float d0, d1;
      unpack_f32x2(fma_f32x2(pack_b32x2(r[j], r[j + 1]), c2, negm2), d0, d1);
      const float e0 = fast_exp2(d0);
      const float e1 = fast_exp2(d1);
      ls2 = add_f32x2(ls2, pack_f32x2(e0, e1));
      r[j] = __float_as_uint(e0);
      r[j + 1] = __float_as_uint(e1);
    }
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int j = 0; j < 16; j += 4) {
      const uint32_t a = split_e4m3x2(pack_b32x2(r[16 * q + j], r[16 * q + j + 1]));
      const uint32_t b = split_e4m3x2(pack_b32x2(r[16 * q + j + 2], r[16 * q + j + 3]));
      hw[j / 4] = (a & 0xFFFFu) | (b << 16);
      lw[j / 4] = (a >> 16) | (b & 0xFFFF0000u);
    }
    st_async_v4(p_dst + q * 128, hw[0], hw[1], hw[2], hw[3], peer_bar);
    st_async_v4(p_dst + (kTile / 16) * 128 + q * 128, lw[0], lw[1], lw[2], lw[3], peer_bar);
  }
  float ls0, ls1;
  unpack_f32x2(ls2, ls0, ls1);
  return ls0 + ls1;
}

// Largest of a tile's 96 raw scores.
MLA_DEVI float tile_max(const uint32_t (&r)[kTile]) {
  float m0 = __uint_as_float(r[0]), m1 = __uint_as_float(r[1]), m2 = __uint_as_float(r[2]);
#pragma unroll
  for (int j = 3; j + 5 < kTile; j += 6) {
    m0 = max3f(m0, __uint_as_float(r[j]), __uint_as_float(r[j + 1]));
    m1 = max3f(m1, __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
    m2 = max3f(m2, __uint_as_float(r[j + 4]), __uint_as_float(r[j + 5]));
  }
  m0 = max3f(m0, m1, m2);
  return max3f(m0, __uint_as_float(r[kTile - 3]), max3f(__uint_as_float(r[kTile - 2]),
                                                      __uint_as_float(r[kTile - 1]), m0));
}

// Softmax warps: one thread per head row (TMEM lane); each warp runs on its
// own (no barrier between the four warps per tile). Per tile: the 96 scores
// are read from tensor memory with one wait, the S buffer is released at
// once, the running row maximum m moves only when the tile's maximum exceeds
// it by more than rescale_threshold (log2 units; always on an item's first
// tile), and one pass writes P and the row record {alpha, l, m} into the
// output CTA with remote stores.
//
// FP8 path: the raw scores carry the row's Q scale 2^k and the cache scale,
// so the multiplier is c = sm_scale * log2(e) * kv_scale * 2^k (2^k read
// from the Q loaders' ring slot of the item at the item's start, before any
// of its S buffers is released: the loaders reuse a slot four items later,
// after the S MMAs of a later tile, which wait for that release). At the
// item's start these warps also convert panels 5..8 of the item's Q (the
// loaders convert 0..4). P is shipped as p' = p * 2^kF8PShift, and the
// record's m is m - kF8PShift, so that lse = m + log2(l) and out = O / l
// hold unchanged.
template <bool F8>
MLA_DEVI void score_softmax(const DecodeParams& p, Ctrl* c, uint8_t* data, uint32_t tmem,
                            int warp, int lane, int it0, int it1) {
  const int row = (warp & 3) * 32 + lane;
  const uint32_t trow = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
  const bool elected = (warp == 2 && lane == 0);
  const float sl2 = p.scale_log2;
  float c_row = sl2;
  int n_items = 0;
  // Peer (output CTA) P buffers, record ring and p_full barriers.
  const uint32_t peer_pbuf0 = map_to_rank(smem_addr(data + kNumVSlots * kVHalfBytes), 1);
  const uint32_t peer_rec0 =
      map_to_rank(smem_addr(data + kNumVSlots * kVHalfBytes + kNumPBufs * kPBytes), 1);
  const uint32_t peer_pfull0 = map_to_rank(smem_addr(&c->p_full[0]), 1);
  // Byte offset of this row inside a P tile (core-matrix row); chunk q adds 128*q.
  const uint32_t prow_off = (row >> 3) * kPGroupBytes + (row & 7) * 16;

  int g = 0;
  bool ok = true;
  int cur = it0;
  while (cur < it1 && tiles_of(item_at(p, cur)) == 0) ++cur;
  while (cur < it1 && ok) {
    const WorkItem w = item_at(p, cur);
    const int nt = tiles_of(w);
    int nxt = cur + 1;
    while (nxt < it1 && tiles_of(item_at(p, nxt)) == 0) ++nxt;
    float m_used = -INFINITY, l = 0.0f;
    const int item = n_items++;
    if constexpr (F8) {
      // The row's Q scale 2^k (the loaders' ring slot of this item), then the
      // second part of the item's Q conversion once the previous item's S
      // MMAs are done with Q.
      const int slot = item % kF8QScaleSlots;
      if (!__all_sync(kFullMask, mbar_wait(smem_addr(&c->qs_ready[slot]),
                                           (item / kF8QScaleSlots) & 1))) {
        ok = false;
        break;
      }
      // (a 32-bit shared-memory address keeps this path within the
      // register budget of the role)
      float qs;
      asm volatile("ld.shared.f32 %0, [%1];" : "=f"(qs)
                   : "r"(smem_addr(data) + kF8NumStages * kF8StageBytes +
                         (slot * kMaxHeads + row) * 4)
                   : "memory");
      c_row = sl2 * p.kv_scale * qs;
      if (item > 0 && !__all_sync(kFullMask, mbar_wait(smem_addr(&c->q_free),
                                                       static_cast<uint32_t>((item - 1) & 1)))) {
        ok = false;
        break;
      }
      tc_after_sync();
      // qs = 2^k exactly, so 2^-k has the exponent field 254 - (k + 127).
      const float inv_s = __uint_as_float((254u << 23) - __float_as_uint(qs));
      if (!convert_q_f8(p, c, w, row, trow, inv_s, kQPanelsByLoader, kNumPanels)) {
        ok = false;
        break;
      }
    }
    for (int i = 0; i < nt; ++i, ++g) {
      const int s = g & 1;
      const int k = g % kNumPBufs;
      const uint32_t ph = static_cast<uint32_t>(g / kNumPBufs) & 1u;   // P buffer use parity
      const uint32_t scol = trow + kTmemS0 + s * kTile;
      // Columns of this row's tile that it attends to (<= 0: none).
      const int valid = min(kTile, row_end(p, w, row) - (w.t0 + i * kTile));
      if (!__all_sync(kFullMask, mbar_wait(smem_addr(&c->s_full[s]), (g >> 1) & 1))) {
        ok = false;
        break;
      }
      if (row == 0) MLA_TRACE_AT(4, g);
      tc_after_sync();
      uint32_t r[kTile];
#pragma unroll
      for (int j = 0; j < kTile; j += 32)
        tmem_ld32(scol + j, *reinterpret_cast<uint32_t(*)[32]>(&r[j]));
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < kTile; j += 8) reg_fence8(&r[j]);
      // The scores are in registers: the S buffer may take tile g + 2.
      tc_before_sync();
      mbar_arrive(smem_addr(&c->s_free[s]));
      if (row == 0) MLA_TRACE_AT(17, g);
      if (valid < kTile) {   // columns past the row's end are -inf
#pragma unroll
        for (int j = 0; j < kTile; ++j) r[j] = j < valid ? r[j] : 0xFF800000u;
      }
      // Lazy rescale: keep the running maximum unless the tile's maximum lies
      // more than the threshold above it (always on an item's first tile,
      // where m is -inf); P rescaled by alpha then reaches the output CTA.
      const float m_tile = tile_max(r) * c_row;
      float alpha = 1.0f;
      if (m_tile > m_used + rescale_threshold<F8>()) {
        alpha = fast_exp2(m_used - m_tile);   // 0 on an item's first tile
        l *= alpha;
        m_used = m_tile;
      }
      // P buffer k may be overwritten once P.V of tile g - 2 has read it
      // (lane 0 waits with cluster acquire; the warp barrier orders the other
      // lanes' remote stores after it).
      if (g >= kNumPBufs) {
        int got = 1;
        if (lane == 0) got = mbar_wait_cluster(smem_addr(&c->p_empty[k]), ph ^ 1u);
        got = __shfl_sync(kFullMask, got, 0);
        __syncwarp();
        if (!got) {
          ok = false;
          break;
        }
      }
      if (row == 0) MLA_TRACE_AT(5, g);
      const uint32_t bar = peer_pfull0 + k * 8;
      // A row that has seen no token yet (m = -inf) writes p = 0.
      const float m_eff = F8 ? m_used - kF8PShift : m_used;
      const float mneg = m_used == -INFINITY ? 0.0f : -m_eff;
      const uint64_t c2 = pack_f32x2(c_row, c_row);
      if (F8)
        l += softmax_tile_f8(r, c2, pack_f32x2(mneg, mneg), peer_pbuf0 + k * kPBytes + prow_off, bar);
      else
        l += softmax_tile(r, c2, pack_f32x2(mneg, mneg), peer_pbuf0 + k * kPBytes + prow_off, bar);
      st_async_v4(peer_rec0 + (g % kNumRecSlots) * kRecBytes + row * 16, __float_as_uint(alpha),
                  __float_as_uint(l), __float_as_uint(m_eff), 0u, bar);
      if (row == 0) MLA_TRACE_AT(6, g);
    }
    cur = nxt;
  }
  // Drain: the peer's last commits (arriving on p_empty) are consumed, so
  // nothing remote is in flight into this CTA when it exits.
  if (elected) {
    if (ok)
      for (int gg = (g > kNumPBufs ? g - kNumPBufs : 0); gg < g; ++gg)
        if (!mbar_wait_cluster(smem_addr(&c->p_empty[gg % kNumPBufs]), (gg / kNumPBufs) & 1)) {
          ok = false;
          break;
        }
  }
  if (!ok && lane == 0) report(p, 4u);
}

// ----------------------------------------------------------- output CTA roles

// TMA producer warp of the output CTA: V into a ring of kNumVSlots 48 KB
// slots. bf16: each tile as two half-tiles of 256 columns (4 panels); FP8:
// each tile's 512 columns in one slot.
template <bool F8>
MLA_DEVI void out_producer(const DecodeParams& p, Ctrl* c, uint8_t* data, int lane, int it0,
                           int it1) {
  constexpr int kParts = F8 ? 1 : 2;   // slots per tile
  uint32_t err = 0;
  const uint64_t policy = policy_evict_first();   // last use of these lines
  int h = 0;
  bool ok = true;
  for (int it = it0; it < it1 && ok; ++it) {
    const WorkItem w = item_at(p, it);
    const int nt = tiles_of(w);
    PageWindow win;
    for (int i = 0; i < nt && ok; ++i) {
      const int tile_t0 = w.t0 + i * kTile;
      const int n = pieces_per_tile(p.block_size);
      int r0, large;
      piece_shape(p.block_size, lane < n ? lane : 0, r0, large);
      window_cover(p, w, tile_t0, win, lane);
      const int y = cache_row(p, w, tile_t0 + r0, win, err);
      for (int half = 0; half < kParts; ++half, ++h) {
        const int v = h % kNumVSlots;
        if (h >= kNumVSlots &&
            !warp_wait(smem_addr(&c->v_empty[v]), ((h / kNumVSlots) - 1) & 1, lane)) {
          ok = false;
          break;
        }
        MLA_TRACE_AT(8 + half, h / kParts);
        const uint32_t full = smem_addr(&c->v_full[v]);
        if (lane == 0) mbar_arrive_expect_tx(full, kVHalfBytes);
        __syncwarp();
        // One warp instruction: lane j loads piece j.
        if (lane < n) {
          if (F8)
            tma_load_4d(smem_addr(data + v * kVHalfBytes) + (r0 >> 3) * kF8NopeGroupBytes,
                        large ? static_cast<const void*>(&p.tmap_k32)
                              : static_cast<const void*>(&p.tmap_k16),
                        0, 0, 0, y >> 3, full, policy);
          else
            tma_load_4d(smem_addr(data + v * kVHalfBytes) + (r0 >> 3) * kVGroupBytes,
                        large ? static_cast<const void*>(&p.tmap_v32)
                              : static_cast<const void*>(&p.tmap_v16),
                        0, 0, half * kVHalfPanels, y >> 3, full, policy);
        }
      }
    }
  }
  if (!ok) err |= 4u;
  err = __reduce_or_sync(kFullMask, err);
  if (lane == 0) report(p, err);
}

// Prefetch warp of the output CTA: walks the pair's tiles kPrefetchTiles
// ahead of the P tiles received so far and issues per-line L2 prefetches
// (load/store path) for the cache pages of those tiles, so the score CTA's
// TMA loads find them in L2. Pages are contiguous blocks of block_size x
// row bytes (1152 bf16, 576 FP8); each page is prefetched once per item.
template <bool ROWS>
MLA_DEVI void out_prefetcher(const DecodeParams& p, Ctrl* c, int lane, int it0, int it1) {
  const char* cache = reinterpret_cast<const char*>(p.kv_cache);
  const int row_bytes = p.kv_fp8 ? kD : kD * 2;
  const int lines = p.block_size * row_bytes / 128;   // block sizes are multiples of 16
  volatile int32_t* seen = &c->p_seen;
  int g = 0;
  for (int it = it0; it < it1; ++it) {
    const WorkItem w = item_at(p, it);
    const int nt = tiles_of(w);
    const int n_pages = (w.t1 + p.block_size - 1) / p.block_size;
    PageWindow win;
    int next_page = w.t0 / p.block_size;
    for (int i = 0; i < nt; ++i, ++g) {
      // Stay at most kPrefetchTiles ahead (bounded wait: about 1 s).
      int ahead_ok = 1;
      if (lane == 0) {
        const long long t0 = clock64();
        while (*seen < g - kPrefetchTiles) {
          if (clock64() - t0 > kWaitLimitCycles) { ahead_ok = 0; break; }
          __nanosleep(200);
        }
      }
      if (!__shfl_sync(kFullMask, ahead_ok, 0)) return;
      if constexpr (ROWS) {   // row-list mode: the tile's rows, each once
        const int oob = static_cast<int>(p.num_blocks * p.block_size);
        const int32_t* rl = p.rows + static_cast<int64_t>(w.b) * p.rows_stride;
        const int lo = w.t0 + i * kTile, end = min(w.t1, lo + kTile);
        for (int t = lo + lane; t < end; t += 32) {
          const int r = __ldg(&rl[t]);
          if (r < 0 || r >= oob) continue;
          const char* base = cache + static_cast<int64_t>(r) * row_bytes;
          for (int k = 0; k < row_bytes; k += 128)
            asm volatile("prefetch.global.L2 [%0];" :: "l"(base + k));
          asm volatile("prefetch.global.L2 [%0];" :: "l"(base + row_bytes - 1));
        }
        continue;
      }
      const int hi = min(n_pages, (min(w.t1, w.t0 + (i + 1) * kTile) + p.block_size - 1) / p.block_size);
      for (; next_page < hi; ++next_page) {
        const int page = next_page;
        if (win.base < 0 || page < win.base || page >= win.base + 32) {
          win.base = page;
          win.val = (page + lane < n_pages)
                        ? __ldg(&p.block_table[static_cast<int64_t>(w.b) * p.max_blocks + page + lane])
                        : -1;
        }
        const int blk = __shfl_sync(kFullMask, win.val, page - win.base);
        if (blk < 0 || static_cast<int64_t>(blk) >= p.num_blocks) continue;
        const char* base = cache + static_cast<int64_t>(blk) * p.block_size * row_bytes;
        for (int ln = lane; ln < lines; ln += 32)
          asm volatile("prefetch.global.L2 [%0];" :: "l"(base + ln * 128));
      }
    }
  }
}

// MMA issuer: O[:, 256*half ...] += P . V_half (5 k-steps of 16 tokens each).
// An item's first tile overwrites O, so it waits for P itself (no rescale is
// due) and, per half, for the epilogue of the previous item to have read
// those columns; later tiles wait for the correction warps' o_ready.
//
// FP8 path: one V slot per tile; per 256-column half, the hi and the lo terms
// of P each take 3 k-steps of 32 tokens (6 MMAs with N = 256).
template <bool F8, bool ROWS>
MLA_DEVI void out_mma(const DecodeParams& p, Ctrl* c, uint8_t* data, uint32_t tmem, int it0,
                      int it1) {
  int g = 0, h = 0, r = 0, n_items = 0;
  bool ok = true;
  uint8_t* pbufs = data + kNumVSlots * kVHalfBytes;
  for (int it = it0; it < it1 && ok; ++it) {
    const WorkItem w = item_at(p, it);
    const int nt = tiles_of(w);
    if (nt == 0) continue;
    const int item = n_items++;
    for (int i = 0; i < nt; ++i, ++g) {
      const int k = g % kNumPBufs;
      // P of this tile arrived through the peer's remote stores, counted on
      // p_full[k]: this thread acquires that phase itself (cluster scope)
      // for every tile, so the stores are visible to it before the proxy
      // fence below. Every tile also waits for all correction warps to have
      // taken it (o_ready; on an item's first tile there is nothing to
      // rescale, but the wait keeps every correction warp within the P ring:
      // P of tile g + kNumPBufs, the next phase of p_full[k], can then not
      // arrive before each of them has seen this phase).
      if (!mbar_wait_cluster(smem_addr(&c->p_full[k]), (g / kNumPBufs) & 1)) { ok = false; break; }
      if (!mbar_wait(smem_addr(&c->o_ready[r % kNumPBufs]), (r / kNumPBufs) & 1)) { ok = false; break; }
      ++r;
      MLA_TRACE_AT(10, g);
      tc_after_sync();
      // P arrived through remote stores (generic proxy); make them visible to
      // the tensor core's reads of shared memory.
      fence_proxy_async_smem();
      // P: no-swizzle K-major; K-adjacent core matrices 128 B apart, row
      // groups kPGroupBytes apart (layout type 0 in bits 61-63).
      const uint32_t pa = smem_addr(pbufs + k * kPBytes);
      uint64_t a0 = static_cast<uint64_t>((pa >> 4) & 0x3FFFu);
      a0 |= static_cast<uint64_t>(128 >> 4) << 16;
      a0 |= static_cast<uint64_t>(kPGroupBytes >> 4) << 32;
      a0 |= static_cast<uint64_t>(1) << 46;
      if (!F8) {
        for (int half = 0; half < 2; ++half, ++h) {
          const int v = h % kNumVSlots;
          if (i == 0 && item > 0 &&
              !mbar_wait(smem_addr(&c->o_drained[half]), (item - 1) & 1)) { ok = false; break; }
          if (!mbar_wait(smem_addr(&c->v_full[v]), (h / kNumVSlots) & 1)) { ok = false; break; }
          MLA_TRACE_AT(11 + half, g);
          tc_after_sync();
          if constexpr (ROWS) fence_proxy_async_smem();
          // V half: MN-major, 128-byte swizzle; 64-column panels 1 KB apart
          // (LBO), 8-token row groups kVGroupBytes apart (SBO); a k-step of
          // 16 tokens is two row groups.
          const uint64_t b0 = smem_desc(smem_addr(data + v * kVHalfBytes), kAtomBytes, kVGroupBytes);
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk) {
            const uint64_t ad = a0 + static_cast<uint64_t>((kk * 256) >> 4);
            const uint64_t bd = b0 + static_cast<uint64_t>((kk * 2 * kVGroupBytes) >> 4);
            mma_ss(tmem + half * 256, ad, bd, kIdescPV, (i > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(smem_addr(&c->v_empty[v]));
        }
      } else {
        const int v = h % kNumVSlots;
        if (!mbar_wait(smem_addr(&c->v_full[v]), (h / kNumVSlots) & 1)) { ok = false; break; }
        ++h;
        tc_after_sync();
        if constexpr (ROWS) fence_proxy_async_smem();
        // V tile: MN-major, 128-byte swizzle; 128-column panels 1 KB apart
        // (LBO), 8-token row groups kF8NopeGroupBytes apart (SBO); a k-step
        // of 32 tokens is four row groups, a 256-column half two panels.
        // P: hi codes in core-matrix columns 0..5, lo codes in 6..11.
        const uint64_t b0 = smem_desc(smem_addr(data + v * kVHalfBytes), kAtomBytes, kF8NopeGroupBytes);
        for (int half = 0; half < 2; ++half) {
          if (i == 0 && item > 0 &&
              !mbar_wait(smem_addr(&c->o_drained[half]), (item - 1) & 1)) { ok = false; break; }
          MLA_TRACE_AT(11 + half, g);
          tc_after_sync();
#pragma unroll
          for (int part = 0; part < 2; ++part)
#pragma unroll
            for (int kk = 0; kk < kTile / 32; ++kk) {
              const uint64_t ad = a0 + static_cast<uint64_t>((part * (kTile / 16) * 128 + kk * 256) >> 4);
              const uint64_t bd =
                  b0 + static_cast<uint64_t>((half * 2 * kAtomBytes + kk * 4 * kF8NopeGroupBytes) >> 4);
              mma_ss_f8(tmem + half * 256, ad, bd, kIdescPV8, (i > 0 || part > 0 || kk > 0) ? 1u : 0u);
            }
        }
        tc_commit(smem_addr(&c->v_empty[v]));
      }
      if (!ok) break;
      tc_commit(smem_addr(&c->o_done[g % kNumPBufs]));
      tc_commit_multicast(smem_addr(&c->p_empty[k]), static_cast<uint16_t>(0x1));
      MLA_TRACE_AT(13, g);
    }
  }
  if (!ok) report(p, 4u);
}

// 64 columns of this thread's O row (two batched tensor-memory loads, one
// wait), scaled by inv_l, to the output row (bf16) or the split partial (fp32).
MLA_DEVI void drain64(const DecodeParams& p, uint32_t taddr, float inv_l, bool to_out,
                      uint16_t* out_row, float* part_row) {
  uint32_t r[64];
  tmem_ld32(taddr, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
  tmem_ld32(taddr + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
  tmem_wait_ld();
  // The loads write r after they issue: pin every use of r below the wait
  // (nothing else orders the arithmetic on r after it).
#pragma unroll
  for (int j = 0; j < 64; j += 8) reg_fence8(&r[j]);
  if (out_row == nullptr && part_row == nullptr) return;
  // Each store instruction writes 32 rows (one per lane), so its cost grows
  // with the rows it touches, not with its bytes: 32-byte stores (whole
  // sectors) take half as many instructions as 16-byte ones.
  if (to_out) {
    if ((reinterpret_cast<uintptr_t>(out_row) & 31u) == 0) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        uint32_t v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
          v[k] = pack_bf16x2(__uint_as_float(r[16 * e + 2 * k]) * inv_l,
                             __uint_as_float(r[16 * e + 2 * k + 1]) * inv_l);
        st_global_v8(out_row + 16 * e, v);
      }
    } else {   // the caller's out is only 16-byte aligned
      uint4* o = reinterpret_cast<uint4*>(out_row);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        uint4 v;
        v.x = pack_bf16x2(__uint_as_float(r[8 * e + 0]) * inv_l, __uint_as_float(r[8 * e + 1]) * inv_l);
        v.y = pack_bf16x2(__uint_as_float(r[8 * e + 2]) * inv_l, __uint_as_float(r[8 * e + 3]) * inv_l);
        v.z = pack_bf16x2(__uint_as_float(r[8 * e + 4]) * inv_l, __uint_as_float(r[8 * e + 5]) * inv_l);
        v.w = pack_bf16x2(__uint_as_float(r[8 * e + 6]) * inv_l, __uint_as_float(r[8 * e + 7]) * inv_l);
        o[e] = v;
      }
    }
  } else {   // the split partials sit in the 256-byte aligned workspace
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      uint32_t v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = __float_as_uint(__uint_as_float(r[8 * e + k]) * inv_l);
      st_global_v8(part_row + 8 * e, v);
    }
  }
}

// Correction + epilogue warps: one thread per head row (TMEM lane). P tiles
// land on p_full, which the elected thread arms two tiles ahead (one phase per
// tile and buffer), so the MMA warp can also wait on it for an item's first
// tile while these warps are still in the previous item's epilogue.
template <bool F8>
MLA_DEVI void out_correct(const DecodeParams& p, Ctrl* c, uint8_t* data, uint32_t tmem, int warp,
                          int lane, int it0, int it1) {
  const int row = (warp & 3) * 32 + lane;
  const uint32_t trow = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
  const bool elected = (warp == 2 && lane == 0);
  const uint8_t* recs = data + kNumVSlots * kVHalfBytes + kNumPBufs * kPBytes;
  int total = 0;
  for (int it = it0; it < it1; ++it) total += tiles_of(item_at(p, it));
  if (elected)
    for (int k = 0; k < kNumPBufs && k < total; ++k)
      mbar_arrive_expect_tx(smem_addr(&c->p_full[k]), kPMsgBytes);
  int g = 0, r = 0;
  bool ok = true;
  for (int it = it0; it < it1 && ok; ++it) {
    const WorkItem w = item_at(p, it);
    const int nt = tiles_of(w);
    const bool active = row < heads_of(p, w);
    const int64_t orow = static_cast<int64_t>(w.b) * p.H + w.h0 + row;
    if (nt == 0) {  // no tokens: out = 0, lse = -inf (a split piece: an empty partial)
      if (active && w.slot < 0) {
        uint4* o = reinterpret_cast<uint4*>(p.out + orow * kDc);
        for (int e = 0; e < kDc / 8; ++e) o[e] = make_uint4(0u, 0u, 0u, 0u);
        p.lse[orow] = -INFINITY;
      } else if (active) {
        p.part_lse[static_cast<int64_t>(w.slot) * p.H + w.h0 + row] = -INFINITY;
      }
      continue;
    }
    float l_fin = 1.0f, m_fin = 0.0f;
    for (int i = 0; i < nt; ++i, ++g) {
      const int k = g % kNumPBufs;
      if (!__all_sync(kFullMask, mbar_wait_cluster(smem_addr(&c->p_full[k]), (g / kNumPBufs) & 1))) {
        ok = false;
        break;
      }
      // The record arrived through the peer's remote stores; order them
      // before this thread's ordinary shared-memory loads of it.
      fence_proxy_async_smem();
      if (row == 0) {
        MLA_TRACE_AT(14, g);
        atomicAdd(&c->p_seen, 1);
      }
      // The record of tile g stays in its slot until tile g + kNumRecSlots,
      // which the peer ships after P.V of tile g + kNumRecSlots - kNumPBufs
      // (at least g + 1) has completed. That P.V waited for these warps to
      // pass its tile (o_ready), after this read of tile g.
      const float4 rec = reinterpret_cast<const float4*>(recs + (g % kNumRecSlots) * kRecBytes)[row];
      const float alpha = active ? rec.x : 1.0f;
      const float lv = rec.y;
      const float mv = rec.z;
      // A non-first tile rescales O when the softmax maximum moved.
      if (i > 0 && __any_sync(kFullMask, alpha != 1.0f)) {
        if (!__all_sync(kFullMask, mbar_wait(smem_addr(&c->o_done[(g - 1) % kNumPBufs]), ((g - 1) / kNumPBufs) & 1))) {
          ok = false;
          break;
        }
        tc_after_sync();
        // tcgen05.st reads its source registers asynchronously: each store
        // completes (wait::st) before the next load may reuse them.
#pragma unroll 1
        for (int cc = 0; cc < kDc / 32; ++cc) {
          uint32_t rr[32];
          tmem_ld32(trow + cc * 32, rr);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; j += 8) reg_fence8(&rr[j]);
#pragma unroll
          for (int j = 0; j < 32; ++j) rr[j] = __float_as_uint(__uint_as_float(rr[j]) * alpha);
          tmem_st32(trow + cc * 32, rr);
          tmem_wait_st();
        }
      }
      tc_before_sync();
      mbar_arrive(smem_addr(&c->o_ready[r % kNumPBufs]));
      ++r;
      // The next phase of this buffer is P of tile g + kNumPBufs.
      if (elected && g + kNumPBufs < total)
        mbar_arrive_expect_tx(smem_addr(&c->p_full[k]), kPMsgBytes);
      if (row == 0) MLA_TRACE_AT(15, g);
      if (i == nt - 1) {
        l_fin = lv;
        m_fin = mv;
      }
    }
    if (!ok) break;
    // Epilogue: O / l -> out (bf16) or the split partial (fp32), one
    // 256-column half at a time; each half is released to the next item's
    // first P.V as soon as it has been read.
    if (!__all_sync(kFullMask, mbar_wait(smem_addr(&c->o_done[(g - 1) % kNumPBufs]), ((g - 1) / kNumPBufs) & 1))) {
      ok = false;
      break;
    }
    tc_after_sync();
    // A row without tokens in this item (possible with several query tokens
    // per request) has l = 0: out = 0 and lse = -inf. An FP8 cache's scale
    // multiplies V here (and K through the softmax multiplier).
    const float inv_l = l_fin > 0.0f ? (F8 ? p.kv_scale : 1.0f) / l_fin : 0.0f;
    const float lse_val = l_fin > 0.0f ? (m_fin + __log2f(l_fin)) * 0.69314718055994531f : -INFINITY;
    const bool to_out = w.slot < 0;
    uint16_t* out_row = (active && to_out) ? p.out + orow * kDc : nullptr;
    float* part_row = (active && !to_out)
                          ? p.part_o + (static_cast<int64_t>(w.slot) * p.H + w.h0 + row) * kDc
                          : nullptr;
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        const int col = half * 256 + cc * 64;
        drain64(p, trow + col, inv_l, to_out, out_row ? out_row + col : nullptr,
                part_row ? part_row + col : nullptr);
      }
      tc_before_sync();
      mbar_arrive(smem_addr(&c->o_drained[half]));
    }
    if (active) {
      if (to_out) p.lse[orow] = lse_val;
      else p.part_lse[static_cast<int64_t>(w.slot) * p.H + w.h0 + row] = lse_val;
    }
  }
  if (!ok) report(p, 4u);
}

// Warm L2 with the Q rows of the pair's first item, at kernel entry: the
// loader warps start only after the prologue's barrier, and their three round
// trips to DRAM otherwise set the start of every pair (about 13 us from launch
// for 128 heads). The calling warp has already arrived on that barrier, so
// the read of the work list here does not delay it. Out of line, so the
// kernel body keeps its code layout.
__device__ __noinline__ void prefetch_first_q(const DecodeParams& p, int it0, int it1) {
  for (int it = it0; it < it1; ++it) {
    const WorkItem w = item_at(p, it);
    if (tiles_of(w) == 0) continue;
    const int64_t qrow = static_cast<int64_t>(w.b) * p.H + w.h0;
    const int nh = heads_of(p, w);
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(p.q_nope + qrow * kDc), "r"(nh * kDc * 2) : "memory");
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(p.q_pe + qrow * kDr), "r"(nh * kDr * 2) : "memory");
    return;
  }
}

template <bool F8, bool ROWS>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
mla_decode_kernel(const __grid_constant__ DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  grid_dep_wait();     // the previous kernel on the stream (e.g. the row lists) is complete
  grid_dep_launch();   // the combine kernel may be scheduled as pairs finish
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Ctrl* c = reinterpret_cast<Ctrl*>(base);
  uint8_t* data = base + kCtrlBytes;
  const uint32_t rank = cluster_rank();
  const int cid = static_cast<int>(cluster_id_x());
  const int it0 = p.cluster_offsets[cid];
  const int it1 = p.cluster_offsets[cid + 1];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < num_stages<F8>(); ++s) {
      mbar_init(smem_addr(&c->kv_full[s]), ROWS ? 32 * kRowsScoreWarps : 1);
      mbar_init(smem_addr(&c->kv_empty[s]), 1);
    }
    for (int j = 0; j < kNumPBufs; ++j) {
      mbar_init(smem_addr(&c->o_ready[j]), 128);
      mbar_init(smem_addr(&c->o_done[j]), 1);
    }
    for (int j = 0; j < 2; ++j) {
      mbar_init(smem_addr(&c->s_full[j]), 1);
      mbar_init(smem_addr(&c->s_free[j]), 128);
      mbar_init(smem_addr(&c->o_drained[j]), 128);
    }
    for (int j = 0; j < kNumPanels; ++j) mbar_init(smem_addr(&c->q_ready[j]), 4);
    mbar_init(smem_addr(&c->q_free), 1);
    for (int k = 0; k < kNumPBufs; ++k) {
      mbar_init(smem_addr(&c->p_empty[k]), 1);
      mbar_init(smem_addr(&c->p_full[k]), 1);
    }
    for (int v = 0; v < kNumVSlots; ++v) {
      mbar_init(smem_addr(&c->v_full[v]), ROWS ? 32 * kRowsOutWarps : 1);
      mbar_init(smem_addr(&c->v_empty[v]), 1);
    }
    for (int j = 0; j < kF8QScaleSlots; ++j) mbar_init(smem_addr(&c->qs_ready[j]), 128);
    c->p_seen = 0;
    fence_barrier_init();
  }
  if (!ROWS && warp == 0 && lane == 0) {   // row-list mode uses no tensor maps
    prefetch_tmap(&p.tmap_k16);
    prefetch_tmap(&p.tmap_k32);
  } else if (!ROWS && warp == 0 && lane == 1) {
    prefetch_tmap(&p.tmap_v16);
    prefetch_tmap(&p.tmap_v32);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(&c->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_before_sync();
  if (rank == 0 && warp == 8) {
    // This warp arrives first: the prefetch (which reads the work list)
    // does not hold up the pair's start.
    cluster_arrive();
    if (lane == 0) prefetch_first_q(p, it0, it1);
    __syncwarp();
    cluster_wait();
  } else {
    cluster_barrier();
  }
  tc_after_sync();
  const uint32_t tmem = c->tmem_base;

  // Row-list mode: the score CTA's warps 0, 6, 7 and the output CTA's
  // warps 0, 7..11 fetch rows (parts 0..kRows*Warps-1).
  if (rank == 0) {
    if (warp == 0) {
      if constexpr (ROWS) rows_producer<F8, false>(p, c, data, lane, 0, kRowsScoreWarps, it0, it1);
      else score_producer<F8>(p, c, data, lane, it0, it1);
    } else if (warp == 1) {
      if (lane == 0) score_mma<F8, ROWS>(p, c, data, tmem, it0, it1);
    } else if (warp < 6) {
      score_softmax<F8>(p, c, data, tmem, warp, lane, it0, it1);
    } else if (warp >= 8) {
      score_qloader<F8>(p, c, data, tmem, warp, lane, it0, it1);
    } else if (ROWS) {
      rows_producer<F8, false>(p, c, data, lane, warp - 5, kRowsScoreWarps, it0, it1);
    }
  } else {
    if (warp == 0) {
      if constexpr (ROWS) rows_producer<F8, true>(p, c, data, lane, 0, kRowsOutWarps, it0, it1);
      else out_producer<F8>(p, c, data, lane, it0, it1);
    } else if (warp == 1) {
      if (lane == 0) out_mma<F8, ROWS>(p, c, data, tmem, it0, it1);
    } else if (warp < 6) {
      out_correct<F8>(p, c, data, tmem, warp, lane, it0, it1);
    } else if (warp == 6) {
      out_prefetcher<ROWS>(p, c, lane, it0, it1);
    } else if (ROWS) {
      rows_producer<F8, true>(p, c, data, lane, warp - 6, kRowsOutWarps, it0, it1);
    }
  }
  __syncwarp();
  tc_before_sync();
  cluster_barrier();
  if (warp == 1) {
    tc_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace
}  // namespace mla
