// C ABI of the paged MLA decode library: the split-KV planner, argument
// checks, the TMA descriptor of the paged cache, and the kernel launches.
//
// The planner is the "tile scheduler" and split-KV choice of "SM100 Cutlass
// MLA decode with unrestricted num_heads (< 128) for DeepSeek TP" (vLLM PR
// #20769, bot summary), sized per decode batch as its review thread asks; the
// workspace it sizes belongs to the caller, who may pass uninitialised memory
// (the same review asks for torch.empty rather than torch.zeros).
#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <new>
#include <queue>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "../../include/mla_decode.h"
#include "mla_internal.h"

using mla::CombineItem;
using mla::WorkItem;

struct mla_plan_s {
  // H: query rows per request (q_len * heads); the kernels and the schedule
  // work in rows, heads and q_len are what the caller passed.
  int B = 0, H = 0, block_size = 0, max_blocks = 0;
  int heads = 0, q_len = 1;
  int device = -1;
  bool host_only = false;
  int num_clusters = 0;                  // CTA pairs the schedule may use
  int num_launch = 0;                    // pairs that hold work items (launched)
  int force_splits = 0;
  bool lengths_are_bounds = false;       // seq_lens are upper bounds; kernels read the true ones
  std::vector<int32_t> seq_lens;
  std::vector<int32_t> splits;           // per request
  std::vector<WorkItem> items;           // grouped by CTA pair
  std::vector<int32_t> item_cluster;     // parallel to items
  std::vector<int32_t> cluster_offsets;  // num_clusters + 1
  std::vector<CombineItem> combine;
  int max_split = 0;                     // largest n_slots over the combine items
  int num_slots = 0;
  size_t workspace_bytes = 0;
  // Device copy of the schedule: [error word | items | offsets | combine].
  uint8_t* d_buf = nullptr;
  size_t d_cap = 0;
  // Pinned staging for asynchronous uploads, two buffers used in turn, each
  // with the event of the last copy that read it.
  uint8_t* h_stage[2] = {nullptr, nullptr};
  size_t h_cap[2] = {0, 0};
  cudaEvent_t upload_done[2] = {nullptr, nullptr};
  int stage_turn = 0;
  // Buffers replaced by a larger one while queued work might still read them;
  // freed by mla_plan_destroy, after its device synchronisation.
  std::vector<uint8_t*> retired_dev;
  std::vector<uint8_t*> retired_host;
  size_t off_items = 0, off_offsets = 0, off_combine = 0, sched_bytes = 0;
  // Cached TMA descriptors (K and V boxes, 16- and 32-row) of the last cache seen.
  CUtensorMap tmap_k16;
  CUtensorMap tmap_k32;
  CUtensorMap tmap_v16;
  CUtensorMap tmap_v32;
  const void* tmap_ptr = nullptr;
  int64_t tmap_blocks = -1;
  int tmap_fp8 = -1;
  // Sparse plans (mla_sparse_plan): the schedule is that of requests of
  // sparse_topk list positions (max_blocks blocks of kSparseBlock); the
  // workspace holds the decode's partials, then at sparse_off the per-request
  // counts of valid entries and the compacted row lists [B, sparse_topk].
  int sparse_topk = 0;
  size_t sparse_off = 0;
};

namespace {

constexpr size_t kErrBytes = 256;
constexpr int kMaxForcedSplits = 4096;

mla_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool device_is_sm103(int dev) {
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
    return false;
  if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return false;
  return major == 10 && minor == 3;
}

// One-time per-device setup (kernel attributes) and the co-resident pair count.
struct DeviceInfo {
  bool prepared = false;
  int clusters = 0;
};
std::mutex g_dev_mu;
DeviceInfo g_dev[64];

mla_status_t prepare_device(int dev, int* clusters) {
  if (dev < 0 || dev >= 64) return MLA_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.prepared) {
    if (!device_is_sm103(dev)) return MLA_ERR_UNSUPPORTED_DEVICE;
    if (mla::decode_prepare_device() != cudaSuccess || mla::combine_prepare_device() != cudaSuccess)
      return MLA_ERR_CUDA;
    int n = 0;
    if (mla::decode_max_clusters(&n) != cudaSuccess || n <= 0) return MLA_ERR_CUDA;
    d.clusters = n;
    d.prepared = true;
  }
  if (clusters) *clusters = d.clusters;
  return MLA_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// ------------------------------------------------------------ the scheduler

struct Piece {
  int b;
  int tile_begin, tile_end;
};

// Split request b's tiles into n near-equal contiguous pieces.
void split_request(int b, int tiles, int n, std::vector<Piece>& out) {
  if (tiles == 0) {
    out.push_back({b, 0, 0});
    return;
  }
  n = std::max(1, std::min(n, tiles));
  const int q = tiles / n, r = tiles % n;
  int t = 0;
  for (int i = 0; i < n; ++i) {
    const int len = q + (i < r ? 1 : 0);
    out.push_back({b, t, t + len});
    t += len;
  }
}

// Longest-processing-time-first assignment; returns the makespan in cost
// units and fills owner[i] with the CTA pair of piece i; order lists the
// pieces longest first.
double lpt(const std::vector<double>& cost, int nc, std::vector<int>* order,
           std::vector<int>* owner) {
  std::vector<int> idx(cost.size());
  for (size_t i = 0; i < idx.size(); ++i) idx[i] = static_cast<int>(i);
  std::stable_sort(idx.begin(), idx.end(), [&](int a, int b) { return cost[a] > cost[b]; });
  using Slot = std::pair<double, int>;
  std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> heap;
  for (int c = 0; c < nc; ++c) heap.push({0.0, c});
  double makespan = 0.0;
  if (owner) owner->assign(cost.size(), 0);
  for (int i : idx) {
    Slot s = heap.top();
    heap.pop();
    s.first += cost[i];
    makespan = std::max(makespan, s.first);
    if (owner) (*owner)[i] = s.second;
    heap.push(s);
  }
  if (order) *order = idx;
  return makespan;
}

// Exchange pass over an assignment. While the most loaded pair can hand an
// item to another pair, or swap it for a smaller item there, so that both end
// below the current makespan, it does so: partner pairs are tried from the
// least loaded up, and with the first partner that admits an improvement the
// exchange leaving the larger of the two loads smallest is made. Returns the
// new makespan.
double refine_assignment(const std::vector<double>& cost, int nc, std::vector<int>& owner) {
  std::vector<double> load(nc, 0.0);
  std::vector<std::vector<int>> held(nc);
  for (size_t i = 0; i < cost.size(); ++i) {
    load[owner[i]] += cost[i];
    held[owner[i]].push_back(static_cast<int>(i));
  }
  std::vector<int> by_load(nc);   // pairs in increasing load
  for (int c = 0; c < nc; ++c) by_load[c] = c;
  auto resort = [&]() {           // insertion sort: at most two pairs moved
    for (int a = 1; a < nc; ++a) {
      const int c = by_load[a];
      int b = a;
      while (b > 0 && load[by_load[b - 1]] > load[c]) {
        by_load[b] = by_load[b - 1];
        --b;
      }
      by_load[b] = c;
    }
  };
  std::sort(by_load.begin(), by_load.end(), [&](int a, int b) { return load[a] < load[b]; });
  constexpr double kEps = 1e-9;
  const int max_rounds = 8 * nc;
  for (int round = 0; round < max_rounds; ++round) {
    const int top = by_load[nc - 1];
    const double lt = load[top];
    int bi = -1, bc = -1, bj = -1;   // item of top, partner pair, item coming back (-1: none)
    for (int k = 0; k < nc - 1 && bi < 0; ++k) {
      const int c = by_load[k];
      const double lc = load[c];
      if (lc + kEps >= lt) break;
      double best = lt - kEps;
      const std::vector<int>& ht = held[top];
      const std::vector<int>& hc = held[c];
      for (size_t a = 0; a < ht.size(); ++a) {
        const double ci = cost[ht[a]];
        const double moved = std::max(lt - ci, lc + ci);
        if (moved < best) { best = moved; bi = static_cast<int>(a); bc = c; bj = -1; }
        for (size_t q = 0; q < hc.size(); ++q) {
          const double d = ci - cost[hc[q]];
          if (d <= 0.0) continue;
          const double swapped = std::max(lt - d, lc + d);
          if (swapped < best) { best = swapped; bi = static_cast<int>(a); bc = c; bj = static_cast<int>(q); }
        }
      }
    }
    if (bi < 0) break;
    const int i = held[top][bi];
    held[top].erase(held[top].begin() + bi);
    load[top] -= cost[i];
    if (bj >= 0) {
      const int j = held[bc][bj];
      held[bc].erase(held[bc].begin() + bj);
      load[bc] -= cost[j];
      held[top].push_back(j);
      load[top] += cost[j];
      owner[j] = top;
    }
    held[bc].push_back(i);
    load[bc] += cost[i];
    owner[i] = bc;
    resort();
  }
  return load[by_load[nc - 1]];
}

// Cost model in units of one 80-token tile of the steady-state pipeline:
//  - every item costs its tiles plus a fixed start/finish overhead (Q load
//    into tensor memory, pipeline fill, epilogue);
//  - every split item also writes an fp32 partial of H x 512 that the
//    combine kernel reads back, spread over all pairs; the combine launch
//    adds a fixed cost when any request is split.
constexpr double kItemOverheadTiles = 2.5;
constexpr double kCombineLaunchTiles = 3.0;

// Partial write and read-back of one split item (its head group's rows).
double split_cost_tiles(int H) {
  const double h = std::min(H, mla::kMaxHeads);
  const double bytes = 2.0 * (h * mla::kDc * 4 + h * 4);
  return bytes / (static_cast<double>(mla::kTile) * mla::kD * 2);
}

int head_groups(int H) { return (H + mla::kMaxHeads - 1) / mla::kMaxHeads; }

void build_schedule(mla_plan_s* p) {
  const int B = p->B;
  std::vector<int> tiles(B);
  int max_tiles = 0;
  for (int b = 0; b < B; ++b) {
    tiles[b] = (p->seq_lens[b] + mla::kTile - 1) / mla::kTile;
    max_tiles = std::max(max_tiles, tiles[b]);
  }
  const int nc = p->num_clusters;
  const double pen = split_cost_tiles(p->H);
  const int ng = head_groups(p->H);   // every KV piece is processed once per head group

  auto make_pieces = [&](int chunk, std::vector<Piece>& pieces) {
    pieces.clear();
    for (int b = 0; b < B; ++b) {
      int n;
      if (p->force_splits > 0) n = std::min(p->force_splits, std::max(tiles[b], 1));
      else n = tiles[b] == 0 ? 1 : (tiles[b] + chunk - 1) / chunk;
      split_request(b, tiles[b], n, pieces);
    }
  };
  // Cost of a candidate under perfect balance: a lower bound on evaluate().
  // It never decreases as the chunks get smaller (more items, more split
  // partials), so the search below stops once it reaches the best cost found.
  auto lower_bound = [&](const std::vector<Piece>& pieces) {
    std::vector<int> count(B, 0);
    for (const Piece& pc : pieces) count[pc.b]++;
    double sum = 0.0;
    int split_items = 0;
    for (const Piece& pc : pieces) {
      sum += ng * ((pc.tile_end - pc.tile_begin) + kItemOverheadTiles);
      if (count[pc.b] > 1) split_items += ng;
    }
    double m = sum / nc;
    if (split_items > 0) m += kCombineLaunchTiles + split_items * pen / nc;
    return m;
  };
  // Items: piece i, head group q -> index i * ng + q.
  auto evaluate = [&](const std::vector<Piece>& pieces, std::vector<int>* order,
                      std::vector<int>* owner) {
    std::vector<double> cost(pieces.size() * ng);
    std::vector<int> count(B, 0);
    for (const Piece& pc : pieces) count[pc.b]++;
    int split_items = 0;
    for (size_t i = 0; i < pieces.size(); ++i) {
      for (int q = 0; q < ng; ++q)
        cost[i * ng + q] = (pieces[i].tile_end - pieces[i].tile_begin) + kItemOverheadTiles;
      if (count[pieces[i].b] > 1) split_items += ng;
    }
    double m = lpt(cost, nc, order, owner);
    if (split_items > 0) m += kCombineLaunchTiles + split_items * pen / nc;
    return m;
  };

  std::vector<Piece> best, cand;
  if (p->force_splits > 0 || max_tiles <= 1) {
    make_pieces(std::max(max_tiles, 1), best);
  } else {
    double best_cost = 0.0;
    int last_chunk = -1;
    for (int k = 1; k <= 256; ++k) {
      const int chunk = std::max(1, (max_tiles + k - 1) / k);
      if (chunk == last_chunk) continue;
      last_chunk = chunk;
      make_pieces(chunk, cand);
      if (cand.size() * ng > static_cast<size_t>(std::max(64 * nc, B * ng))) break;
      if (!best.empty() && lower_bound(cand) >= best_cost - 1e-9) break;
      const double c = evaluate(cand, nullptr, nullptr);
      if (best.empty() || c < best_cost - 1e-9) {
        best_cost = c;
        best = cand;
      }
      if (chunk == 1) break;
    }
  }
  std::vector<int> order, owner;
  evaluate(best, &order, &owner);
  {
    std::vector<double> cost(best.size() * ng);
    for (size_t i = 0; i < cost.size(); ++i)
      cost[i] = (best[i / ng].tile_end - best[i / ng].tile_begin) + kItemOverheadTiles;
    refine_assignment(cost, nc, owner);
  }

  // Slots for split pieces, combine list, per-request split counts.
  std::vector<int> count(B, 0);
  for (const Piece& pc : best) count[pc.b]++;
  p->splits.assign(B, 0);
  p->max_split = 0;
  std::vector<int> first_slot(B, -1);
  int slots = 0;
  p->combine.clear();
  for (int b = 0; b < B; ++b) {
    p->splits[b] = count[b];
    if (count[b] > 1) {
      first_slot[b] = slots;
      p->combine.push_back({b, slots, count[b], 0});
      slots += count[b];
      p->max_split = std::max(p->max_split, count[b]);
    }
  }
  // A split piece owns one partial slot, shared by its head groups (each
  // writes its own heads' rows).
  std::vector<int> next_slot = first_slot;
  std::vector<WorkItem> piece_item(best.size() * ng);
  for (size_t i = 0; i < best.size(); ++i) {
    const Piece& pc = best[i];
    WorkItem w{};
    w.b = pc.b;
    w.t0 = pc.tile_begin * mla::kTile;
    w.t1 = std::min(pc.tile_end * mla::kTile, p->seq_lens[pc.b]);
    w.slot = count[pc.b] > 1 ? next_slot[pc.b]++ : -1;
    w.seq_len = p->seq_lens[pc.b];
    for (int q = 0; q < ng; ++q) {
      w.h0 = q * mla::kMaxHeads;
      piece_item[i * ng + q] = w;
    }
  }
  // Group by pair, each pair's list in assignment order (longest first).
  // Pairs left without items are dropped, so only pairs with work launch.
  std::vector<std::vector<int>> per(nc);
  for (int i : order) per[owner[i]].push_back(i);
  p->items.clear();
  p->item_cluster.clear();
  p->cluster_offsets.clear();
  for (int c = 0; c < nc; ++c) {
    if (per[c].empty()) continue;
    const int launched = static_cast<int>(p->cluster_offsets.size());
    p->cluster_offsets.push_back(static_cast<int32_t>(p->items.size()));
    for (int i : per[c]) {
      p->items.push_back(piece_item[i]);
      p->item_cluster.push_back(launched);
    }
  }
  p->num_launch = static_cast<int>(p->cluster_offsets.size());
  p->cluster_offsets.push_back(static_cast<int32_t>(p->items.size()));
  p->num_slots = slots;
  const size_t o_bytes = static_cast<size_t>(slots) * p->H * mla::kDc * 4;
  const size_t l_bytes = static_cast<size_t>(slots) * p->H * 4;
  p->workspace_bytes = slots ? align_up(align_up(o_bytes, 256) + l_bytes, 256) : 0;

  p->off_items = kErrBytes;
  p->off_offsets = align_up(p->off_items + p->items.size() * sizeof(WorkItem), 16);
  p->off_combine = align_up(p->off_offsets + p->cluster_offsets.size() * 4, 16);
  p->sched_bytes = align_up(p->off_combine + p->combine.size() * sizeof(CombineItem), 256);
}

mla_status_t check_plan_args(int B, int H, const int32_t* seq_lens, int block_size,
                             int max_blocks, int q_len = 1) {
  if (B < 1 || H < 1 || q_len < 1 || !seq_lens || max_blocks < 1) return MLA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(H) * q_len > mla::kMaxPlanHeads) return MLA_ERR_INVALID_ARG;
  if (block_size != 16 && block_size != 32 && block_size != 64 && block_size != 128)
    return MLA_ERR_INVALID_ARG;
  const int64_t cap = static_cast<int64_t>(max_blocks) * block_size;
  if (cap >= (int64_t{1} << 30)) return MLA_ERR_INVALID_ARG;
  for (int b = 0; b < B; ++b) {
    if (seq_lens[b] < 0 || seq_lens[b] > cap) return MLA_ERR_INVALID_ARG;
    // Several query tokens are the request's last tokens: it holds them all.
    if (q_len > 1 && seq_lens[b] != 0 && seq_lens[b] < q_len) return MLA_ERR_INVALID_ARG;
  }
  return MLA_OK;
}

// Copy the schedule to the device: synchronously (plan creation) or as an
// asynchronous copy on `stream` from pinned staging (mla_plan_update). The
// asynchronous path never waits for the device: a device buffer that must
// grow is replaced, the error word is carried over by a copy ordered on the
// stream, and the old buffer is kept until the plan is destroyed; the two
// staging buffers alternate, so a copy from one may still be queued while the
// other is filled.
mla_status_t upload(mla_plan_s* p, cudaStream_t stream, bool sync) {
  if (p->host_only) return MLA_OK;
  if (p->sched_bytes > p->d_cap) {
    const size_t cap = align_up(p->sched_bytes * 2, 4096);
    uint8_t* nb = nullptr;
    if (cudaMalloc(&nb, cap) != cudaSuccess) return MLA_ERR_CUDA;
    cudaError_t e;
    if (p->d_buf) {
      // The error word is sticky until mla_check_device_error: carry it over.
      e = sync ? cudaMemcpy(nb, p->d_buf, kErrBytes, cudaMemcpyDeviceToDevice)
               : cudaMemcpyAsync(nb, p->d_buf, kErrBytes, cudaMemcpyDeviceToDevice, stream);
      p->retired_dev.push_back(p->d_buf);
    } else {
      e = cudaMemset(nb, 0, kErrBytes);
    }
    p->d_buf = nb;
    p->d_cap = cap;
    if (e != cudaSuccess) return MLA_ERR_CUDA;
  }
  const int k = p->stage_turn;
  p->stage_turn ^= 1;
  if (!p->upload_done[k] &&
      cudaEventCreateWithFlags(&p->upload_done[k], cudaEventDisableTiming) != cudaSuccess)
    return MLA_ERR_CUDA;
  // This staging buffer may still feed the copy before last.
  if (cudaEventSynchronize(p->upload_done[k]) != cudaSuccess) return MLA_ERR_CUDA;
  if (p->sched_bytes > p->h_cap[k]) {
    if (p->h_stage[k]) p->retired_host.push_back(p->h_stage[k]);
    p->h_stage[k] = nullptr;
    p->h_cap[k] = 0;
    const size_t cap = align_up(p->sched_bytes * 2, 4096);
    if (cudaMallocHost(&p->h_stage[k], cap) != cudaSuccess) return MLA_ERR_CUDA;
    p->h_cap[k] = cap;
  }
  uint8_t* h = p->h_stage[k];
  std::memcpy(h + p->off_items, p->items.data(), p->items.size() * sizeof(WorkItem));
  std::memcpy(h + p->off_offsets, p->cluster_offsets.data(), p->cluster_offsets.size() * 4);
  std::memcpy(h + p->off_combine, p->combine.data(), p->combine.size() * sizeof(CombineItem));
  const size_t n = p->sched_bytes - kErrBytes;
  if (sync) {
    if (cudaMemcpy(p->d_buf + kErrBytes, h + kErrBytes, n, cudaMemcpyHostToDevice) != cudaSuccess)
      return MLA_ERR_CUDA;
  } else {
    if (cudaMemcpyAsync(p->d_buf + kErrBytes, h + kErrBytes, n, cudaMemcpyHostToDevice, stream) !=
        cudaSuccess)
      return MLA_ERR_CUDA;
  }
  if (cudaEventRecord(p->upload_done[k], sync ? nullptr : stream) != cudaSuccess) return MLA_ERR_CUDA;
  return MLA_OK;
}

void free_plan(mla_plan_s* p) {
  if (!p) return;
  if (p->d_buf || !p->retired_dev.empty()) {
    cudaDeviceSynchronize();
    if (p->d_buf) cudaFree(p->d_buf);
    for (uint8_t* b : p->retired_dev) cudaFree(b);
  }
  for (int k = 0; k < 2; ++k) {
    if (p->upload_done[k]) {
      cudaEventSynchronize(p->upload_done[k]);
      cudaEventDestroy(p->upload_done[k]);
    }
    if (p->h_stage[k]) cudaFreeHost(p->h_stage[k]);
  }
  for (uint8_t* b : p->retired_host) cudaFreeHost(b);
  delete p;
}

bool aligned(const void* ptr, size_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

// Tensor maps of the cache at kv_cache, kept in the plan until the cache
// pointer, pool size or element type changes.
// bf16: the cache is viewed as a 4-D tensor {64 columns, 8 rows, 9 panels,
// row groups of 8} with strides of 1152 B (row), 128 B (panel) and 9216 B
// (row group), so one box brings a run of 16 or 32 rows across several
// panels and lands as [row group][panel][8 rows][128 B] (128-byte swizzle,
// zero fill outside the pool). Boxes: 2 or min(block_size, 32)/8 row groups;
// 9 panels (K: all 576 columns) or 4 panels (one half of V).
// FP8: columns 0..511 as {128 columns, 8 rows, 4 panels, row groups}
// (strides 576, 128, 4608 B; 128-byte swizzle), the K and V boxes; columns
// 512..575 as {64 columns, 8 rows, row groups} (strides 576, 4608 B; 64-byte
// swizzle), the rope boxes. Splitting the row keeps every box inside it: a
// 128-column view of the rope columns would read 64 bytes past each row,
// and past the pool's end on its last row.
mla_status_t refresh_kv_maps(mla_plan_s* p, const void* kv_cache, int64_t num_blocks, bool fp8) {
  if (p->tmap_ptr == kv_cache && p->tmap_blocks == num_blocks && p->tmap_fp8 == (fp8 ? 1 : 0))
    return MLA_OK;
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return MLA_ERR_CUDA;
  p->tmap_ptr = nullptr;
  const cuuint64_t groups = static_cast<cuuint64_t>(num_blocks) * p->block_size / 8;
  const int large = std::min(p->block_size, mla::kRowsLargeBox);
  const cuuint32_t g_small = mla::kRowsSmallBox / 8, g_large = static_cast<cuuint32_t>(large / 8);
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  if (!fp8) {
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(mla::kPanelCols), 8,
                                static_cast<cuuint64_t>(mla::kNumPanels), groups};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(mla::kD) * 2,
                                   static_cast<cuuint64_t>(mla::kPanelCols) * 2,
                                   static_cast<cuuint64_t>(mla::kD) * 2 * 8};
    CUtensorMap* maps[4] = {&p->tmap_k16, &p->tmap_k32, &p->tmap_v16, &p->tmap_v32};
    const cuuint32_t box_groups[4] = {g_small, g_large, g_small, g_large};
    const int panels[4] = {mla::kNumPanels, mla::kNumPanels, mla::kVHalfPanels, mla::kVHalfPanels};
    for (int i = 0; i < 4; ++i) {
      const cuuint32_t box[4] = {static_cast<cuuint32_t>(mla::kPanelCols), 8,
                                 static_cast<cuuint32_t>(panels[i]), box_groups[i]};
      if (enc(maps[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(kv_cache), dims,
              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return MLA_ERR_INVALID_ARG;
    }
  } else {
    const cuuint64_t dims[4] = {128, 8, static_cast<cuuint64_t>(mla::kF8Panels), groups};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(mla::kD), 128,
                                   static_cast<cuuint64_t>(mla::kD) * 8};
    CUtensorMap* maps[2] = {&p->tmap_k16, &p->tmap_k32};
    const cuuint32_t box_groups[2] = {g_small, g_large};
    for (int i = 0; i < 2; ++i) {
      const cuuint32_t box[4] = {128, 8, static_cast<cuuint32_t>(mla::kF8Panels), box_groups[i]};
      if (enc(maps[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(kv_cache), dims,
              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return MLA_ERR_INVALID_ARG;
    }
    const cuuint64_t rdims[3] = {static_cast<cuuint64_t>(mla::kDr), 8, groups};
    const cuuint64_t rstrides[2] = {static_cast<cuuint64_t>(mla::kD),
                                    static_cast<cuuint64_t>(mla::kD) * 8};
    CUtensorMap* rmaps[2] = {&p->tmap_v16, &p->tmap_v32};
    void* rope = const_cast<uint8_t*>(static_cast<const uint8_t*>(kv_cache) + mla::kDc);
    for (int i = 0; i < 2; ++i) {
      const cuuint32_t box[3] = {static_cast<cuuint32_t>(mla::kDr), 8, box_groups[i]};
      if (enc(rmaps[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, rope, rdims, rstrides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return MLA_ERR_INVALID_ARG;
    }
  }
  p->tmap_ptr = kv_cache;
  p->tmap_blocks = num_blocks;
  p->tmap_fp8 = fp8 ? 1 : 0;
  return MLA_OK;
}

}  // namespace

extern "C" {

mla_status_t mla_decode_plan_ex(int B, int H, const int32_t* seq_lens_host, int block_size,
                                int max_blocks, const mla_plan_options_t* opts,
                                mla_plan_t* plan_out) {
  if (!plan_out) return MLA_ERR_INVALID_ARG;
  *plan_out = nullptr;
  mla_plan_options_t o{};
  if (opts) o = *opts;
  if (o.q_len < 0) return MLA_ERR_INVALID_ARG;
  const int q_len = o.q_len > 0 ? o.q_len : 1;
  mla_status_t st = check_plan_args(B, H, seq_lens_host, block_size, max_blocks, q_len);
  if (st != MLA_OK) return st;
  if (o.num_clusters < 0 || o.force_splits < 0 || o.force_splits > kMaxForcedSplits)
    return MLA_ERR_INVALID_ARG;
  mla_plan_s* p = new (std::nothrow) mla_plan_s();
  if (!p) return MLA_ERR_INVALID_ARG;
  p->B = B;
  p->H = H * q_len;
  p->heads = H;
  p->q_len = q_len;
  p->block_size = block_size;
  p->max_blocks = max_blocks;
  p->host_only = o.host_only != 0;
  p->force_splits = o.force_splits;
  p->lengths_are_bounds = o.lengths_are_bounds != 0;
  p->seq_lens.assign(seq_lens_host, seq_lens_host + B);
  if (!p->host_only || o.num_clusters == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
      free_plan(p);
      return MLA_ERR_UNSUPPORTED_DEVICE;
    }
    int clusters = 0;
    st = prepare_device(dev, &clusters);
    if (st != MLA_OK) {
      free_plan(p);
      return st;
    }
    p->device = dev;
    p->num_clusters = o.num_clusters > 0 ? std::min(o.num_clusters, clusters) : clusters;
  } else {
    p->num_clusters = o.num_clusters;
  }
  build_schedule(p);
  st = upload(p, nullptr, true);
  if (st != MLA_OK) {
    free_plan(p);
    return st;
  }
  *plan_out = p;
  return MLA_OK;
}

mla_status_t mla_decode_plan(int B, int H, const int32_t* seq_lens_host, int block_size,
                             int max_blocks, mla_plan_t* plan_out) {
  return mla_decode_plan_ex(B, H, seq_lens_host, block_size, max_blocks, nullptr, plan_out);
}

mla_status_t mla_plan_update(mla_plan_t p, const int32_t* seq_lens_host, void* stream) {
  if (!p || p->sparse_topk > 0) return MLA_ERR_INVALID_ARG;
  mla_status_t st =
      check_plan_args(p->B, p->heads, seq_lens_host, p->block_size, p->max_blocks, p->q_len);
  if (st != MLA_OK) return st;
  if (!p->host_only) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != p->device) return MLA_ERR_INVALID_ARG;
  }
  p->seq_lens.assign(seq_lens_host, seq_lens_host + p->B);
  build_schedule(p);
  return upload(p, static_cast<cudaStream_t>(stream), false);
}

size_t mla_plan_workspace_bytes(mla_plan_t p) { return p ? p->workspace_bytes : 0; }

int mla_plan_num_splits(mla_plan_t p, int b) {
  if (!p || b < 0 || b >= p->B) return -1;
  return p->splits[b];
}

int mla_plan_num_work_items(mla_plan_t p) { return p ? static_cast<int>(p->items.size()) : -1; }

int mla_plan_num_clusters(mla_plan_t p) { return p ? p->num_launch : -1; }

int mla_plan_work_item_heads(mla_plan_t p, int i, int32_t* h_begin, int32_t* h_end) {
  if (!p || i < 0 || i >= static_cast<int>(p->items.size())) return -1;
  const WorkItem& w = p->items[i];
  if (h_begin) *h_begin = w.h0;
  if (h_end) *h_end = std::min(p->H, w.h0 + mla::kMaxHeads);
  return 0;
}

int mla_plan_work_item(mla_plan_t p, int i, int32_t* b, int32_t* t0, int32_t* t1, int32_t* slot,
                       int32_t* cluster) {
  if (!p || i < 0 || i >= static_cast<int>(p->items.size())) return -1;
  const WorkItem& w = p->items[i];
  if (b) *b = w.b;
  if (t0) *t0 = w.t0;
  if (t1) *t1 = w.t1;
  if (slot) *slot = w.slot;
  if (cluster) *cluster = p->item_cluster[i];
  return 0;
}

}  // extern "C"

namespace {

// mla_decode and mla_decode_fp8: the same launches on a bf16 (fp8 = false)
// or an E4M3 cache with per-tensor scale kv_scale.
mla_status_t decode_impl(mla_plan_t p, const void* q_nope, const void* q_pe, const void* kv_cache,
                         bool fp8, float kv_scale, int64_t num_blocks, const int32_t* block_table,
                         const int32_t* seq_lens, float sm_scale, void* out, float* lse,
                         void* workspace, size_t workspace_bytes, void* stream,
                         const int32_t* rows = nullptr, int64_t num_rows = 0) {
  // rows != null: row-list mode (sparse plans only); token t of request b is
  // cache row rows[b * sparse_topk + t] of num_rows; the block table is unused.
  const bool sparse = rows != nullptr;
  if (!p || p->host_only || (p->sparse_topk > 0) != sparse) return MLA_ERR_INVALID_ARG;
  if (fp8 && (!(kv_scale > 0.0f) || !std::isfinite(kv_scale))) return MLA_ERR_INVALID_ARG;
  if (!q_nope || !q_pe || !kv_cache || (!block_table && !sparse) || !seq_lens || !out || !lse)
    return MLA_ERR_INVALID_ARG;
  if (!aligned(q_nope, 16) || !aligned(q_pe, 16) || !aligned(kv_cache, 16) || !aligned(out, 16) ||
      !aligned(lse, 4) || !aligned(block_table, 4) || !aligned(seq_lens, 4))
    return MLA_ERR_INVALID_ARG;
  const int64_t cache_rows = sparse ? num_rows : num_blocks * p->block_size;
  if (num_blocks < 1 || cache_rows < 1 || cache_rows + 64 >= (int64_t{1} << 31))
    return MLA_ERR_INVALID_ARG;
  if (!(sm_scale > 0.0f) || !std::isfinite(sm_scale)) return MLA_ERR_INVALID_ARG;
  const size_t ws_need = sparse ? p->sparse_off : p->workspace_bytes;   // the decode's own part
  if (ws_need > 0) {
    if (!workspace || workspace_bytes < ws_need) return MLA_ERR_WORKSPACE_TOO_SMALL;
    if (!aligned(workspace, 256)) return MLA_ERR_INVALID_ARG;
  }
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_UNSUPPORTED_DEVICE;
  if (dev != p->device) return MLA_ERR_INVALID_ARG;
  mla_status_t st = prepare_device(dev, nullptr);
  if (st != MLA_OK) return st;

  if (!sparse) {   // row-list mode reads rows with plain copies, not tensor maps
    st = refresh_kv_maps(p, kv_cache, num_blocks, fp8);
    if (st != MLA_OK) return st;
  }

  mla::DecodeParams dp;
  std::memset(&dp, 0, sizeof(dp));
  if (!sparse) {
    dp.tmap_k16 = p->tmap_k16;
    dp.tmap_k32 = p->tmap_k32;
    dp.tmap_v16 = p->tmap_v16;
    dp.tmap_v32 = p->tmap_v32;
  }
  dp.kv_cache = kv_cache;
  dp.q_nope = static_cast<const uint16_t*>(q_nope);
  dp.q_pe = static_cast<const uint16_t*>(q_pe);
  dp.block_table = block_table;
  dp.seq_lens = seq_lens;
  dp.out = static_cast<uint16_t*>(out);
  dp.lse = lse;
  const size_t o_bytes = static_cast<size_t>(p->num_slots) * p->H * mla::kDc * 4;
  dp.part_o = static_cast<float*>(workspace);
  dp.part_lse = p->num_slots
                    ? reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + align_up(o_bytes, 256))
                    : nullptr;
  dp.items = reinterpret_cast<const WorkItem*>(p->d_buf + p->off_items);
  dp.cluster_offsets = reinterpret_cast<const int32_t*>(p->d_buf + p->off_offsets);
  dp.err = reinterpret_cast<uint32_t*>(p->d_buf);
  dp.H = p->H;
  dp.q_len = p->q_len;
  dp.heads = p->heads;
  // Row-list mode views the cache as blocks of one row.
  dp.block_size = sparse ? 1 : p->block_size;
  dp.max_blocks = p->max_blocks;
  dp.num_blocks = sparse ? num_rows : num_blocks;
  dp.rows = rows;
  dp.rows_stride = sparse ? p->sparse_topk : 0;
  dp.scale_log2 = sm_scale * 1.4426950408889634f;
  dp.dynamic_lens = p->lengths_are_bounds ? 1 : 0;
  dp.kv_fp8 = fp8 ? 1 : 0;
  dp.kv_scale = fp8 ? kv_scale : 1.0f;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (mla::launch_decode(dp, p->num_launch, s) != cudaSuccess) return MLA_ERR_CUDA;
  if (!p->combine.empty()) {
    mla::CombineParams cp;
    cp.items = reinterpret_cast<const CombineItem*>(p->d_buf + p->off_combine);
    cp.part_o = dp.part_o;
    cp.part_lse = dp.part_lse;
    cp.out = dp.out;
    cp.lse = lse;
    cp.H = p->H;
    if (mla::launch_combine(cp, static_cast<int>(p->combine.size()), p->max_split, s) !=
        cudaSuccess)
      return MLA_ERR_CUDA;
  }
  return MLA_OK;
}

}  // namespace

extern "C" {

mla_status_t mla_decode(mla_plan_t p, const void* q_nope, const void* q_pe, const void* kv_cache,
                        int64_t num_blocks, const int32_t* block_table, const int32_t* seq_lens,
                        float sm_scale, void* out, float* lse, void* workspace,
                        size_t workspace_bytes, void* stream) {
  return decode_impl(p, q_nope, q_pe, kv_cache, false, 1.0f, num_blocks, block_table, seq_lens,
                     sm_scale, out, lse, workspace, workspace_bytes, stream);
}

mla_status_t mla_decode_fp8(mla_plan_t p, const void* q_nope, const void* q_pe,
                            const void* kv_cache_fp8, float kv_scale, int64_t num_blocks,
                            const int32_t* block_table, const int32_t* seq_lens, float sm_scale,
                            void* out, float* lse, void* workspace, size_t workspace_bytes,
                            void* stream) {
  return decode_impl(p, q_nope, q_pe, kv_cache_fp8, true, kv_scale, num_blocks, block_table,
                     seq_lens, sm_scale, out, lse, workspace, workspace_bytes, stream);
}

mla_status_t mla_sparse_plan(int B, int H, int topk, const mla_plan_options_t* opts,
                             mla_plan_t* plan_out) {
  if (!plan_out) return MLA_ERR_INVALID_ARG;
  *plan_out = nullptr;
  if (B < 1 || topk < 1 || topk > (1 << 20)) return MLA_ERR_INVALID_ARG;
  mla_plan_options_t o{};
  if (opts) o = *opts;
  if (o.q_len > 1) return MLA_ERR_INVALID_ARG;   // one selection per request: one query token
  o.lengths_are_bounds = 1;
  const int max_blocks_c = (topk + mla::kSparseBlock - 1) / mla::kSparseBlock;
  std::vector<int32_t> bounds(B, topk);
  mla_status_t st = mla_decode_plan_ex(B, H, bounds.data(), mla::kSparseBlock, max_blocks_c, &o,
                                       plan_out);
  if (st != MLA_OK) return st;
  mla_plan_s* p = *plan_out;
  p->sparse_topk = topk;
  p->sparse_off = align_up(p->workspace_bytes, 256);
  p->workspace_bytes = p->sparse_off + align_up(static_cast<size_t>(B) * 4, 256) +
                       static_cast<size_t>(B) * topk * 4;
  return MLA_OK;
}

mla_status_t mla_decode_sparse(mla_plan_t p, const void* q_nope, const void* q_pe,
                               const void* kv_cache, int kv_fp8, float kv_scale,
                               int64_t num_blocks, int block_size, const int32_t* block_table,
                               int max_blocks, const int32_t* seq_lens,
                               const int32_t* topk_indices, float sm_scale, void* out, float* lse,
                               void* workspace, size_t workspace_bytes, void* stream) {
  if (!p || p->host_only || p->sparse_topk <= 0) return MLA_ERR_INVALID_ARG;
  if (!kv_cache || !block_table || !seq_lens || !topk_indices) return MLA_ERR_INVALID_ARG;
  if (kv_fp8 != 0 && kv_fp8 != 1) return MLA_ERR_INVALID_ARG;
  if (!aligned(kv_cache, 16) || !aligned(block_table, 4) || !aligned(seq_lens, 4) ||
      !aligned(topk_indices, 4))
    return MLA_ERR_INVALID_ARG;
  if (block_size != 16 && block_size != 32 && block_size != 64 && block_size != 128)
    return MLA_ERR_INVALID_ARG;
  // Rows are int32 TMA coordinates.
  if (max_blocks < 1 || num_blocks < 1 || num_blocks * block_size + 64 >= (int64_t{1} << 31))
    return MLA_ERR_INVALID_ARG;
  // What the decode step checks, checked before the row-list kernel runs.
  if (!q_nope || !q_pe || !out || !lse || !aligned(q_nope, 16) || !aligned(q_pe, 16) ||
      !aligned(out, 16) || !aligned(lse, 4))
    return MLA_ERR_INVALID_ARG;
  if (!(sm_scale > 0.0f) || !std::isfinite(sm_scale)) return MLA_ERR_INVALID_ARG;
  if (kv_fp8 && (!(kv_scale > 0.0f) || !std::isfinite(kv_scale))) return MLA_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < p->workspace_bytes) return MLA_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned(workspace, 256)) return MLA_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_UNSUPPORTED_DEVICE;
  if (dev != p->device) return MLA_ERR_INVALID_ARG;
  mla_status_t st = prepare_device(dev, nullptr);
  if (st != MLA_OK) return st;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* counts = reinterpret_cast<int32_t*>(ws + p->sparse_off);
  int32_t* rows = reinterpret_cast<int32_t*>(ws + p->sparse_off + align_up(p->B * 4, 256));
  mla::SparseRowsParams rp;
  rp.num_blocks = num_blocks;
  rp.block_size = block_size;
  rp.max_blocks = max_blocks;
  rp.block_table = block_table;
  rp.seq_lens = seq_lens;
  rp.topk_indices = topk_indices;
  rp.topk = p->sparse_topk;
  rp.rows = rows;
  rp.counts = counts;
  rp.err = reinterpret_cast<uint32_t*>(p->d_buf);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (mla::launch_sparse_rows(rp, p->B, s) != cudaSuccess) return MLA_ERR_CUDA;
  return decode_impl(p, q_nope, q_pe, kv_cache, kv_fp8 != 0, kv_scale, num_blocks, nullptr, counts,
                     sm_scale, out, lse, workspace, p->sparse_off, stream, rows,
                     num_blocks * block_size);
}

// The allocation-free variant: the workspace and the device copy of the work
// list are carved from the library's fixed device scratch
// (mla_no_alloc_sm103.cu) instead of caller or plan memory; the error word is
// the caller's. Layout of the scratch per call: [unused 256 B | work list as
// laid out by build_schedule | split partials o | split partials lse].
mla_status_t mla_decode_no_alloc(mla_plan_t p, const void* q_nope, const void* q_pe,
                                 const void* kv_cache, int64_t num_blocks,
                                 const int32_t* block_table, const int32_t* seq_lens,
                                 float sm_scale, void* out, float* lse, uint32_t* err_bits,
                                 void* stream) {
  if (!p || p->sparse_topk > 0) return MLA_ERR_INVALID_ARG;
  if (!q_nope || !q_pe || !kv_cache || !block_table || !seq_lens || !out || !lse || !err_bits)
    return MLA_ERR_INVALID_ARG;
  if (!aligned(q_nope, 16) || !aligned(q_pe, 16) || !aligned(kv_cache, 16) || !aligned(out, 16) ||
      !aligned(lse, 4) || !aligned(block_table, 4) || !aligned(seq_lens, 4) ||
      !aligned(err_bits, 4))
    return MLA_ERR_INVALID_ARG;
  if (num_blocks < 1 || num_blocks * p->block_size + 64 >= (int64_t{1} << 31))
    return MLA_ERR_INVALID_ARG;
  if (!(sm_scale > 0.0f) || !std::isfinite(sm_scale)) return MLA_ERR_INVALID_ARG;
  // Schedule and partials must fit the fixed scratch; checked before any
  // device call so that an oversize plan is refused the same way everywhere.
  const size_t o_bytes = static_cast<size_t>(p->num_slots) * p->H * mla::kDc * 4;
  if (p->sched_bytes + p->workspace_bytes > mla::kNoAllocScratchBytes)
    return MLA_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The work list is copied from the plan's host vectors. Under stream
  // capture such a copy would become a graph node that reads those vectors
  // at every replay, after a later mla_plan_update or mla_plan_destroy may
  // have reallocated or freed them, so a capturing stream is refused, before
  // any other CUDA call (some would invalidate the caller's capture).
  cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &capture) != cudaSuccess) return MLA_ERR_CUDA;
  if (capture != cudaStreamCaptureStatusNone) return MLA_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_UNSUPPORTED_DEVICE;
  if (p->device >= 0 && dev != p->device) return MLA_ERR_INVALID_ARG;
  mla_status_t st = prepare_device(dev, nullptr);
  if (st != MLA_OK) return st;
  uint8_t* scratch = nullptr;
  if (mla::no_alloc_scratch(dev, &scratch) != cudaSuccess) return MLA_ERR_CUDA;
  st = refresh_kv_maps(p, kv_cache, num_blocks, false);
  if (st != MLA_OK) return st;

  // The caller's error word is the only state that must start at zero: the
  // work list is rewritten below, and every partial slot is written in full
  // by its work item before the combine kernel reads it.
  uint32_t* err = err_bits;
  if (cudaMemsetAsync(err, 0, sizeof(uint32_t), s) != cudaSuccess) return MLA_ERR_CUDA;
  // Outside capture, a copy from pageable memory has been staged by the time
  // cudaMemcpyAsync returns, so a later mla_plan_update cannot change what
  // this call reads.
  if (cudaMemcpyAsync(scratch + p->off_items, p->items.data(), p->items.size() * sizeof(WorkItem),
                      cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(scratch + p->off_offsets, p->cluster_offsets.data(),
                      p->cluster_offsets.size() * sizeof(int32_t), cudaMemcpyHostToDevice,
                      s) != cudaSuccess)
    return MLA_ERR_CUDA;
  if (!p->combine.empty() &&
      cudaMemcpyAsync(scratch + p->off_combine, p->combine.data(),
                      p->combine.size() * sizeof(CombineItem), cudaMemcpyHostToDevice,
                      s) != cudaSuccess)
    return MLA_ERR_CUDA;

  uint8_t* ws = scratch + p->sched_bytes;  // sched_bytes is a multiple of 256
  mla::DecodeParams dp;
  std::memset(&dp, 0, sizeof(dp));
  dp.tmap_k16 = p->tmap_k16;
  dp.tmap_k32 = p->tmap_k32;
  dp.tmap_v16 = p->tmap_v16;
  dp.tmap_v32 = p->tmap_v32;
  dp.kv_cache = kv_cache;
  dp.q_nope = static_cast<const uint16_t*>(q_nope);
  dp.q_pe = static_cast<const uint16_t*>(q_pe);
  dp.block_table = block_table;
  dp.seq_lens = seq_lens;
  dp.out = static_cast<uint16_t*>(out);
  dp.lse = lse;
  dp.part_o = p->num_slots ? reinterpret_cast<float*>(ws) : nullptr;
  dp.part_lse = p->num_slots ? reinterpret_cast<float*>(ws + align_up(o_bytes, 256)) : nullptr;
  dp.items = reinterpret_cast<const WorkItem*>(scratch + p->off_items);
  dp.cluster_offsets = reinterpret_cast<const int32_t*>(scratch + p->off_offsets);
  dp.err = err;
  dp.H = p->H;
  dp.q_len = p->q_len;
  dp.heads = p->heads;
  dp.block_size = p->block_size;
  dp.max_blocks = p->max_blocks;
  dp.num_blocks = num_blocks;
  dp.scale_log2 = sm_scale * 1.4426950408889634f;
  dp.dynamic_lens = p->lengths_are_bounds ? 1 : 0;
  if (mla::launch_decode(dp, p->num_launch, s) != cudaSuccess) return MLA_ERR_CUDA;
  if (!p->combine.empty()) {
    mla::CombineParams cp;
    cp.items = reinterpret_cast<const CombineItem*>(scratch + p->off_combine);
    cp.part_o = dp.part_o;
    cp.part_lse = dp.part_lse;
    cp.out = dp.out;
    cp.lse = lse;
    cp.H = p->H;
    if (mla::launch_combine(cp, static_cast<int>(p->combine.size()), p->max_split, s) !=
        cudaSuccess)
      return MLA_ERR_CUDA;
  }
  return MLA_OK;
}

mla_status_t mla_check_device_error(mla_plan_t p, void* stream, uint32_t* bits_out) {
  if (bits_out) *bits_out = 0;
  if (!p || p->host_only || !p->d_buf) return MLA_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MLA_ERR_CUDA;
  uint32_t bits = 0;
  if (cudaMemcpy(&bits, p->d_buf, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return MLA_ERR_CUDA;
  if (bits && cudaMemset(p->d_buf, 0, 4) != cudaSuccess) return MLA_ERR_CUDA;
  if (bits_out) *bits_out = bits;
  return bits ? MLA_ERR_DEVICE_FAULT : MLA_OK;
}

void mla_plan_destroy(mla_plan_t p) { free_plan(p); }

const char* mla_status_string(mla_status_t s) {
  switch (s) {
    case MLA_OK: return "ok";
    case MLA_ERR_INVALID_ARG: return "invalid argument";
    case MLA_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs sm_103)";
    case MLA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MLA_ERR_CUDA: return "CUDA runtime error";
    case MLA_ERR_DEVICE_FAULT: return "device reported bad input";
  }
  return "unknown status";
}

int mla_device_supported(void) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  return device_is_sm103(dev) ? 1 : 0;
}

mla_status_t mla_selftest_wait_timeout(void* stream, uint32_t* bits_out) {
  if (!bits_out) return MLA_ERR_INVALID_ARG;
  *bits_out = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || !device_is_sm103(dev)) return MLA_ERR_UNSUPPORTED_DEVICE;
  uint32_t* word = nullptr;
  if (cudaMalloc(&word, sizeof(uint32_t)) != cudaSuccess) return MLA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  mla_status_t st = MLA_OK;
  if (cudaMemsetAsync(word, 0, sizeof(uint32_t), s) != cudaSuccess ||
      mla::launch_wait_timeout_selftest(word, s) != cudaSuccess ||
      cudaMemcpyAsync(bits_out, word, sizeof(uint32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    st = MLA_ERR_CUDA;
  cudaFree(word);
  return st;
}

}  // extern "C"
