// Internal types shared by the planner, the C ABI layer and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

namespace mla {

constexpr int kDc = 512;                 // latent c_kv columns (= V width)
constexpr int kDr = 64;                  // rope k_pe columns
constexpr int kD = kDc + kDr;            // 576 bf16 per cached token row
constexpr int kMaxHeads = 128;           // MMA M: one head group; fewer heads are padded inside the kernel
constexpr int kMaxPlanHeads = 1024;      // query heads per request: up to 8 head groups
constexpr int kTile = 96;                // tokens per KV tile (MMA N of the score product)
constexpr int kRowsSmallBox = 16;        // TMA box heights: 16 rows (block size 16) and
constexpr int kRowsLargeBox = 32;        // 32 rows (block sizes >= 32), never crossing a page
constexpr int kMaxPieces = kTile / kRowsSmallBox;      // at most 6 boxes per tile
constexpr int kPanelCols = 64;           // bf16 columns of one 128-byte swizzle panel
constexpr int kNumPanels = kD / kPanelCols;            // 9 panels per row
constexpr int kPanelBytes = kTile * 128;               // one panel of one tile: 12 KB
// Score stage: [row group (12)][panel (9)][8 rows][128 B]; 8-row atoms are
// kKGroupBytes apart along the rows and 1 KB apart along the panels.
constexpr int kStageBytes = kNumPanels * kPanelBytes;  // full 576-wide tile: 108 KB
constexpr int kVHalfPanels = 4;                        // V half = 256 columns
// V half slot: [row group (12)][panel (4)][8 rows][128 B].
constexpr int kVHalfBytes = kVHalfPanels * kPanelBytes;  // 48 KB
constexpr int kAtomBytes = 8 * 128;                      // 8 rows x 128 B (one swizzle atom)
constexpr int kKGroupBytes = kNumPanels * kAtomBytes;    // 9216: row-group stride of a stage
constexpr int kVGroupBytes = kVHalfPanels * kAtomBytes;  // 4096: row-group stride of a V slot
constexpr int kNumStages = 2;            // score CTA: KV tiles in flight
constexpr int kNumVSlots = 3;            // output CTA: V half-tiles in flight
// P tiles in flight (output CTA buffers).
constexpr int kNumPBufs = 3;
// P [128 rows x 96 tokens] bf16 in the no-swizzle K-major layout of 8-row x
// 16-byte core matrices: [row/8][token/8][row%8][16 B]; K-adjacent cores are
// 128 B apart, row groups 1536 B apart. The score CTA's softmax threads write
// it straight into the output CTA's buffer (asynchronous remote stores).
constexpr int kPCoreK = kTile / 8;                     // 12 core matrices along K
constexpr int kPGroupBytes = kPCoreK * 128;            // 1536
constexpr int kPBytes = kMaxHeads / 8 * kPGroupBytes;  // 24 KB
// Row record per tile: {alpha, l, m, 0} as 16 bytes per row.
constexpr int kRecBytes = kMaxHeads * 16;              // 2 KB
constexpr int kPMsgBytes = kPBytes + kRecBytes;        // 26 KB of remote stores per tile
// The output CTA receives P in kNumPBufs buffers and the row record in a ring
// of kNumRecSlots, so a record outlives the reuse of its P buffer.
constexpr int kNumRecSlots = 4;
static_assert(kNumRecSlots >= kNumPBufs + 1, "a record must outlive the reuse of its P buffer");
// FP8 (E4M3) cache: 576-byte rows. Score stage: columns 0..511 as
// [row group (12)][panel (4)][8 rows][128 B] with the 128-byte swizzle, then
// columns 512..575 as [row group (12)][8 rows][64 B] with the 64-byte
// swizzle (two TMA boxes per page piece, so no box reads past a row's end).
// The output CTA loads the same 512-column layout as one V tile per slot.
constexpr int kF8Panels = 4;                                  // 128-column panels of c_kv
constexpr int kF8NopeGroupBytes = kF8Panels * 8 * 128;        // 4096: row-group stride
constexpr int kF8NopeBytes = kTile / 8 * kF8NopeGroupBytes;   // 48 KB
constexpr int kF8RopeGroupBytes = 8 * 64;                     // 512
constexpr int kF8RopeBytes = kTile / 8 * kF8RopeGroupBytes;   // 6 KB
constexpr int kF8StageBytes = kF8NopeBytes + kF8RopeBytes;    // 54 KB
constexpr int kF8NumStages = 4;                               // score CTA: KV tiles in flight
// Per-row scales of the FP8 Q split (Q = 2^k_row (hi + lo)): a ring of
// kF8QScaleSlots items, 128 fp32 each, written by the Q loaders.
constexpr int kF8QScaleSlots = 4;
constexpr int kF8ScoreDataBytes = kF8NumStages * kF8StageBytes + kF8QScaleSlots * kMaxHeads * 4;
static_assert(kF8NopeBytes == 48 * 1024, "an FP8 V tile fills one V slot");
// Q in tensor memory for the FP8 path: hi codes in columns [0, 144), lo
// codes in [144, 288), four E4M3 values per 32-bit column.
constexpr int kF8QLoCol = kD / 4;        // 144

constexpr int kThreads = 384;            // 12 warps per CTA
constexpr int kTmemCols = 512;
// Score CTA TMEM columns: Q (576 bf16 packed in pairs) then two S buffers.
constexpr int kTmemQ = 0;
constexpr int kTmemS0 = kD / 2;          // 288
static_assert(kTmemS0 + 2 * kTile <= kTmemCols, "Q and two S buffers must fit in tensor memory");
// Shared-memory data region (after the 1 KB control block).
constexpr int kCtrlBytes = 1024;
constexpr int kScoreDataBytes = kNumStages * kStageBytes;                            // 216 KB
constexpr int kOutDataBytes =
    kNumVSlots * kVHalfBytes + kNumPBufs * kPBytes + kNumRecSlots * kRecBytes;      // 200 KB
constexpr int kDataBytes0 = kScoreDataBytes > kOutDataBytes ? kScoreDataBytes : kOutDataBytes;
constexpr int kDataBytes = kDataBytes0 > kF8ScoreDataBytes ? kDataBytes0 : kF8ScoreDataBytes;
constexpr int kSmemBytes = kCtrlBytes + kDataBytes + 1024;  // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");

// One unit of work: tokens [t0, t1) of request b. slot >= 0 means the result
// is a split partial written to the workspace; -1 writes out/lse directly.
struct WorkItem {
  int32_t b;
  int32_t t0;
  int32_t t1;
  int32_t slot;
  int32_t seq_len;   // the plan's length of request b (checked against device seq_lens)
  int32_t h0;        // first query row of the item's head group (a multiple of 128)
  int32_t len;       // the request's length in this call (set on the device)
  int32_t pad;
};
static_assert(sizeof(WorkItem) == 32, "WorkItem layout");

// Requests whose KV was split: merge n partial slots starting at first_slot.
struct CombineItem {
  int32_t b;
  int32_t first_slot;
  int32_t n_slots;
  int32_t pad;
};

struct DecodeParams {
  // bf16 cache: 4-D views {64 columns, 8 rows, 9 panels, row groups of 8}
  // (strides: row 1152 B, panel 128 B, row group 9216 B). One box brings a
  // page-aligned run of 16 or 32 rows (2 or 4 row groups) across several
  // 64-column panels and lands in shared memory as [row group][panel][8 rows]
  // [128 B] with the 128-byte swizzle: every 8-row x 128-byte atom of a tile
  // sits at (row group * panels + panel) * 1 KB, whichever page it came from.
  // FP8 cache: tmap_k16/k32 view columns 0..511 as {128 columns, 8 rows,
  // 4 panels, row groups} (strides 576, 128, 4608 B; boxes {128, 8, 4, 2|4},
  // 128-byte swizzle), used for K by the score CTA and for V by the output
  // CTA; tmap_v16/v32 view columns 512..575 as {64 columns, 8 rows, row
  // groups} (strides 576, 4608 B; boxes {64, 8, 2|4}, 64-byte swizzle).
  CUtensorMap tmap_k16;           // box {64, 8, 9, 2}: all 576 columns
  CUtensorMap tmap_k32;           // box {64, 8, 9, 4} (block_size >= 32)
  CUtensorMap tmap_v16;           // box {64, 8, 4, 2}: one 256-column half of V
  CUtensorMap tmap_v32;           // box {64, 8, 4, 4} (block_size >= 32)
  const void* kv_cache;           // the cache itself, for L2 line prefetches
  const uint16_t* q_nope;         // [B, H, 512]
  const uint16_t* q_pe;           // [B, H, 64]
  const int32_t* block_table;     // [B, max_blocks]
  const int32_t* seq_lens;        // [B] device copy
  uint16_t* out;                  // [B, H, 512]
  float* lse;                     // [B, H]
  float* part_o;                  // [slots, H, 512]
  float* part_lse;                // [slots, H]
  const WorkItem* items;          // grouped by CTA pair
  const int32_t* cluster_offsets; // [num_clusters + 1]
  uint32_t* err;                  // device error word
  int H;                          // query rows per request: q_len * heads
  int q_len;                      // query tokens per request (1: plain decode)
  int heads;                      // query heads per token
  int block_size;
  int max_blocks;
  int64_t num_blocks;
  float scale_log2;               // sm_scale * log2(e)
  int dynamic_lens;               // 1: planned lengths are upper bounds; items end at the device length
  int kv_fp8;                     // 1: the cache holds E4M3 bytes [num_blocks, bs, 576]
  float kv_scale;                 // FP8 cache: element value = kv_scale * e4m3(byte)
  // Row-list mode (sparse decode; the kernel's row-list instances): token t
  // of request b is cache row rows[b * rows_stride + t] (row = block id *
  // block_size + slot, with block_size 1 and num_blocks the row count in
  // this mode); the block table and the tensor maps are not used: the rows
  // are copied with 16-byte cp.async into the layout the TMA boxes produce.
  const int32_t* rows;
  int rows_stride;
};

struct CombineParams {
  const CombineItem* items;
  const float* part_o;
  const float* part_lse;
  uint16_t* out;
  float* lse;
  int H;
};

// Sparse (top-k) decode, first step (mla_sparse_sm103.cu): per request, the
// cache rows of the valid list entries, compacted in list order, and their
// count; the decode kernel then runs in row-list mode over them.
struct SparseRowsParams {
  int64_t num_blocks;
  int block_size;
  int max_blocks;
  const int32_t* block_table;     // [B, max_blocks]
  const int32_t* seq_lens;        // [B]
  const int32_t* topk_indices;    // [B, topk]
  int topk;
  int32_t* rows;                  // [B, topk]: rows[b][0..count) written
  int32_t* counts;                // [B]
  uint32_t* err;
};

// Nominal block size of a sparse plan's schedule: the lists are scheduled
// as requests of topk tokens over blocks of this many list positions.
constexpr int kSparseBlock = 64;

// Launch configuration shared by the library's kernels: each is launched as
// a programmatic dependent of the kernel before it on the stream, so its
// launch overlaps that kernel's tail; every kernel waits for its
// prerequisites (griddepcontrol.wait) before it touches global memory.
inline cudaLaunchConfig_t dependent_launch(dim3 grid, dim3 block, size_t smem,
                                           cudaStream_t stream, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// Launchers (defined in the .cu files).
cudaError_t launch_sparse_rows(const SparseRowsParams& p, int B, cudaStream_t stream);
cudaError_t launch_decode(const DecodeParams& p, int num_clusters, cudaStream_t stream);
// The row-list instances (mla_decode_rows_sm103.cu); launch_decode forwards
// a DecodeParams with rows set.
cudaError_t launch_decode_rows(const DecodeParams& p, int num_clusters, cudaStream_t stream);
cudaError_t decode_rows_prepare_device();
// max_slots: the largest n_slots of the combine items (at most 4096).
cudaError_t launch_combine(const CombineParams& p, int num_items, int max_slots,
                           cudaStream_t stream);
cudaError_t combine_prepare_device();
cudaError_t decode_max_clusters(int* num_clusters);
cudaError_t decode_prepare_device();
// One-warp kernel whose wait on a barrier nothing completes must time out
// (sets MLA_DEVERR_TIMEOUT in *err).
cudaError_t launch_wait_timeout_selftest(uint32_t* err, cudaStream_t stream);

// Bytes of the fixed device scratch behind mla_decode_no_alloc.
constexpr size_t kNoAllocScratchBytes = size_t{32} << 20;
// Device address of that scratch on `device`, which must be current; looked
// up on the first call per device and cached (mla_no_alloc_sm103.cu).
cudaError_t no_alloc_scratch(int device, uint8_t** ptr);

}  // namespace mla
