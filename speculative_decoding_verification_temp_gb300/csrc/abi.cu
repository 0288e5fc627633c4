// C ABI of libspecverify: argument checks, workspace layout, launch planning.
// The operations themselves are documented in include/specverify.h.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstddef>
#include <cstdint>

#include "ops.cuh"
#include "precise.cuh"
#include "specverify.h"
#include "verify_units.cuh"

namespace sv {
cudaError_t launch_units(const Params &P, int esize, bool vec, int n_units, size_t smem,
                         cudaStream_t stream);
cudaError_t launch_residual(const Params &P, int esize, float *out, cudaStream_t stream);
cudaError_t launch_tree_mask(const int32_t *parent, int T, int N, int max_depth, uint64_t *mask,
                             int32_t *position, uint32_t *flags, cudaStream_t stream);
cudaError_t launch_stream(const Params &P, int esize, size_t smem, cudaStream_t stream);
cudaError_t launch_first_child(const int32_t *parent, int T, int N, int32_t *first_child,
                               cudaStream_t stream);
cudaError_t launch_refine(const Params &P, int esize, const Exp2Table &tab, cudaStream_t stream);
cudaError_t launch_overlap(const void *target, long long ld_t, const void *draft, long long ld_d,
                           int esize, int B, int gamma, int V, const float *Tp, const float *Tq,
                           float *out_beta, uint32_t *out_flags, cudaStream_t stream);
cudaError_t launch_tree_rerank(const int32_t *parent, const float *confidence, int T, int N, int m,
                               int32_t *out_nodes, int32_t *out_parent, float *out_value,
                               int32_t *out_count, uint32_t *out_flags, cudaStream_t stream);
size_t typical_workspace_bytes(int B, int gamma, int V, int esize);
cudaError_t launch_typical(const void *target, long long ld_t, int esize, int B, int gamma, int V,
                           const float *Tp, const int32_t *tokens, float epsilon, float delta,
                           int32_t *out_num, int32_t *out_tokens, uint32_t *out_flags,
                           void *workspace, cudaStream_t stream);
cudaError_t launch_chain(const Params &P, int esize, const Exp2Table &tab, size_t smem,
                         cudaStream_t stream);
cudaError_t launch_tree_walk(const Params &P, int esize, size_t smem, cudaStream_t stream);
size_t chain_rows_ctl_bytes();
int chain_records_per_chunk();
bool set_profile_events(void *start, void *stop);
}  // namespace sv

namespace {

constexpr int kMaxGamma = 4095;
constexpr int kMaxNodes = 4096;
constexpr size_t kSmemTarget = 72 * 1024;  // three clusters' CTAs per SM
constexpr size_t kSmemHard = 227 * 1024;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Plan {
  int cluster;
  int slice;
  size_t data_off;
  size_t hist_off;
  size_t mass_off;
  size_t smem;
};

// Smallest cluster whose CTAs hold their slice of a target+draft row pair in
// shared memory within the occupancy target; the largest cluster otherwise.
bool make_plan(long long V, int esize, size_t extra, bool topk, bool topp, Plan &pl) {
  pl.data_off = align_up(sizeof(sv::Ctl), 128);
  for (int C = 1; C <= sv::kMaxCluster; C *= 2) {
    const long long slice = static_cast<long long>(align_up(static_cast<size_t>((V + C - 1) / C), 8));
    const size_t data = 2 * static_cast<size_t>(slice) * esize;
    const size_t region = align_up(data > extra ? data : extra, 128);
    const size_t hist = topk ? align_up(sizeof(sv::TopkScratch), 16) : 0;
    const size_t smem = pl.data_off + region + hist + (topp ? sizeof(sv::MassScratch) : 0);
    if (smem <= kSmemTarget || (C == sv::kMaxCluster && smem <= kSmemHard)) {
      pl.cluster = C;
      pl.slice = static_cast<int>(slice);
      pl.hist_off = topk ? pl.data_off + region : 0;
      pl.mass_off = topp ? pl.data_off + region + hist : 0;
      pl.smem = smem;
      return true;
    }
  }
  return false;
}

// Streaming kernel: a unit's rows are cut into slices of at most 32 KB (the
// tasks), streamed through a ring of four slots of at most 16 KB per CTA.
struct StreamPlan {
  int slices;
  int slice;
  int slot_bytes;
  int chunks;
  int ring;
  size_t data_off;
  size_t smem;
};

bool make_stream_plan(long long V, int esize, StreamPlan &sp) {
  constexpr size_t kSlot = 16 * 1024;
  for (int C = 1; C <= 64; C *= 2) {
    const size_t slice = align_up(static_cast<size_t>((V + C - 1) / C), 8);
    const size_t sb = slice * esize;
    if (sb > 2 * kSlot) continue;
    const size_t chunks = (sb + kSlot - 1) / kSlot;
    const size_t slot = ((sb / 16 + chunks - 1) / chunks) * 16;
    sp.slices = C;
    sp.slice = static_cast<int>(slice);
    sp.slot_bytes = static_cast<int>(slot > 16 ? slot : 16);
    sp.chunks = static_cast<int>(chunks);
    sp.ring = 4;  // a weight task holds both rows' chunks at once: ring >= 2 * chunks
    if (sp.ring < 2 * sp.chunks) return false;
    sp.data_off = align_up(sizeof(sv::Ctl3), 128);
    sp.smem = sp.data_off + static_cast<size_t>(sp.ring) * sp.slot_bytes;
    return true;
  }
  return false;
}

// Workspace layout.  The regions that must read zero when the kernels start
// (arrival counters, the weight-task queue and its counters) come first and
// are cleared by every call; everything after them is written before it is
// read within a call.
// Chain path (rows kernel -> draw kernel -> precise kernel): 32 KB chunks
// through a ring of two slots (three rows-kernel CTAs per SM); every row's
// chunks leave one record per consumer warp; the draw works in 256-entry
// steps, whose sums the draw and precise kernels keep in shared memory (4 and
// 16 bytes a step: at most kPassMaxSteps).
struct PassPlan {
  int chunk_elems;
  int cpr;
  int steps;
  int ring;
  int slot_bytes;
};

constexpr int kPassMaxGamma = 31;
constexpr long long kPassMaxSteps = 8192;  // V <= 2,097,152

bool make_pass_plan(long long V, int esize, int gamma, PassPlan &pp) {
  if (gamma > kPassMaxGamma || esize <= 0) return false;
  const long long steps = (V + 255) / 256;
  if (steps > kPassMaxSteps) return false;
  pp.slot_bytes = 32 * 1024;
  pp.ring = 2;  // three CTAs of the rows kernel per SM
  pp.chunk_elems = pp.slot_bytes / esize;
  pp.cpr = static_cast<int>((V + pp.chunk_elems - 1) / pp.chunk_elems);
  pp.steps = static_cast<int>(steps);
  return true;
}

// 64-bit records the chain rows kernel writes for B sequences of gamma drafts
// (one per consumer warp per chunk; 0 when the chain path cannot run the shape).
long long pass_records(long long B, int gamma, long long V, int esize) {
  PassPlan pp{};
  if (!make_pass_plan(V, esize, gamma, pp)) return 0;
  return B * (2 * gamma + 1) * static_cast<long long>(pp.cpr) * sv::chain_records_per_chunk();
}

// 64-bit records the rows kernel writes for T trees of N nodes on the tree
// walk path (N target and N draft rows a tree; 0 when the walk cannot run the
// shape).
long long walk_records(long long T, long long N, long long V, int esize) {
  PassPlan pp{};
  if (N > sv::kWalkMaxNodes || !make_pass_plan(V, esize, 0, pp)) return 0;
  return T * 2 * N * static_cast<long long>(pp.cpr) * sv::chain_records_per_chunk();
}

// 512-entry blocks of a row (the filter kernel's candidates).
long long pass_blocks(long long V) { return (V + 511) / 512; }

// Bytes of the chain path's filter data for B sequences: the rows' block
// maxima (element type) and one (threshold, S) pair per row; 0 when the chain
// path cannot run the shape.
size_t pass_filter_bytes(long long B, int gamma, long long V, int esize) {
  PassPlan pp{};
  if (!make_pass_plan(V, esize, gamma, pp)) return 0;
  const long long rows = B * (2 * gamma + 1);
  return static_cast<size_t>(rows * pass_blocks(V) * esize) + 256 +
         static_cast<size_t>(rows) * sizeof(float2);
}

struct Layout {
  size_t wq_ctr, counters, unit_done, w_done, wq, srec, err, pctr, pseq, near_list, bmax, frec,
      zero_bytes;
  size_t outs, stats, final_unit, first_child, refine, rpart, rc, partials, dstate, wpart, wblk, total;
  long long wq_cap;
};

constexpr long long kMaxSliceBlocks = 2 * 16 + 1;

// slices: slices per unit of the streaming kernel, 0 when only the resident
// kernel can run the shape; recs: records of the chain path (0 when it cannot
// run the shape); fbytes: its filter data (pass_filter_bytes).
Layout layout(long long nseq, long long units, long long slices, long long recs,
              size_t fbytes) {
  Layout L;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, 256);
    return at;
  };
  // A call runs either the streaming kernel or the chain path (or neither):
  // their own regions share addresses, the workspace holds the larger set.
  // zero prefix, common part
  // [0] queue head, [1] tail, [2] units done, [3] refines, [4] redraw barrier
  L.wq_ctr = take(8 * sizeof(uint32_t));
  L.counters = take(static_cast<size_t>(nseq) * sizeof(uint32_t));
  L.err = take(sizeof(uint32_t));
  L.pctr = take(4 * sizeof(uint32_t));  // chain path: precise redraws queued
  // zero prefix, streaming kernel
  L.unit_done = take(static_cast<size_t>(slices ? units : 0) * sizeof(uint32_t));
  L.w_done = take(static_cast<size_t>(slices ? units : 0) * sizeof(uint32_t));
  // weight-task queue: a tree of N nodes runs at most (N - 1) + 2N weight
  // rounds in all (one per rejected child, plus a degenerate fallback and the
  // final draw at each node), one entry per slice
  L.wq_cap = 3 * units * slices;
  L.wq = take(static_cast<size_t>(L.wq_cap) * sizeof(int4));
  L.zero_bytes = off;
  // common
  L.outs = take(static_cast<size_t>(units) * sizeof(sv::UnitOut));
  L.stats = take(static_cast<size_t>(units) * sizeof(sv::UnitStats));
  L.final_unit = take(static_cast<size_t>(nseq) * sizeof(int32_t));
  L.first_child = take(static_cast<size_t>(units) * sizeof(int32_t));
  L.refine = take(static_cast<size_t>(nseq) * sizeof(int4));
  L.rpart = take(static_cast<size_t>(std::max<long long>(sv::kRefineMaxGrid, nseq)) *
                 sizeof(sv::RefinePart));
  L.rc = take(static_cast<size_t>(nseq) * sizeof(double));
  const size_t base = off;
  // streaming kernel
  L.partials = take(static_cast<size_t>(units * slices * 2) * sizeof(sv::SlicePartial));
  L.dstate = take(static_cast<size_t>(slices ? units : 0) * sizeof(sv::DrawState));
  L.wpart = take(static_cast<size_t>(units * slices) * sizeof(float));
  L.wblk = take(static_cast<size_t>(units * slices * kMaxSliceBlocks) * sizeof(float));
  const size_t end_stream = off;
  // chain path: the records, written by the rows kernel before the draw
  // kernel reads them; the queue of precise redraws, written by the draw
  // kernel before the precise kernel reads it
  off = base;
  const long long qseqs = recs ? nseq : 0;
  L.srec = take(static_cast<size_t>(recs) * sizeof(unsigned long long));
  L.pseq = take(static_cast<size_t>(qseqs) * sizeof(sv::PassSeq));
  L.near_list = take(static_cast<size_t>(qseqs) * sizeof(int32_t));
  L.bmax = take(fbytes);  // block maxima, then the per-row filter records
  L.frec = L.bmax;
  L.total = std::max(off, end_stream);
  return L;
}

// Slices of the streaming plan for rows of V entries (0: no streaming plan).
long long stream_slices(long long V, int esize) {
  StreamPlan sp;
  return esize > 0 && make_stream_plan(V, esize, sp) ? sp.slices : 0;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 2^(j/64) as double-float pairs, for the precise redraw.
const sv::Exp2Table &exp2_table() {
  static const sv::Exp2Table tab = [] {
    sv::Exp2Table t;
    for (int j = 0; j < 64; ++j) {
      const double v = std::exp2(j / 64.0);
      t.hi[j] = static_cast<float>(v);
      t.lo[j] = static_cast<float>(v - static_cast<double>(t.hi[j]));
    }
    return t;
  }();
  return tab;
}

spec_status map_cuda(cudaError_t e) { return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA; }

// Cycles the chain rows kernel's first wait on a chunk may take (see
// spec_set_wait_limit); the full bound unless a caller shortened it.
std::atomic<long long> g_first_wait{sv::kWaitLimitCycles};

int esize_of(spec_dtype d) { return d == SPEC_BF16 ? 2 : (d == SPEC_F32 ? 4 : 0); }

// Shared launch path of the chain and tree verifiers.  16-byte aligned rows
// take the streaming chain path (chains of gamma <= 31 and V <= 2,097,152:
// the rows, filter (with a top-k, top-p or min-p array), draw and precise
// kernels) or the tree walk path (trees of at most 256 nodes without a row
// filter, V <= 2,097,152: the first-child, rows, walk and refine kernels);
// aligned rows without filters of larger trees and longer chains the
// streaming kernel; everything else the resident kernel.
spec_status run_units(sv::Params &P, int esize, long long n_units, size_t extra,
                      float *out_residual, void *workspace, size_t workspace_bytes,
                      cudaStream_t stream, bool need_draft_rows) {
  // off the chain path, top-k, top-p and min-p filters run on the resident kernel
  const bool topp = P.pp != nullptr || P.pq != nullptr;
  const bool topk = P.kp != nullptr || P.kq != nullptr || topp || P.mp != nullptr ||
                    P.mq != nullptr;
  const bool vec = aligned16(P.target) && (P.ld_t * esize) % 16 == 0 &&
                   (!need_draft_rows || (aligned16(P.draft) && (P.ld_d * esize) % 16 == 0));
  StreamPlan sp;
  PassPlan pp{};
  Plan pl;
  const bool pass = vec && P.mode == sv::kModeChain &&
                    make_pass_plan(P.V, esize, P.gamma, pp) &&
                    static_cast<long long>(P.nseq) * (2 * P.gamma + 1) * pp.cpr < 0x7FFFFFFFll;
  // trees of at most kWalkMaxNodes nodes without a row filter: the rows
  // stream and the tree walk
  const bool walk = vec && P.mode == sv::kModeTree && !topk && P.ups <= sv::kWalkMaxNodes &&
                    make_pass_plan(P.V, esize, 0, pp) &&
                    static_cast<long long>(P.nseq) * 2 * P.ups * pp.cpr < 0x7FFFFFFFll;
  const bool streaming = !pass && !walk && vec && !topk && make_stream_plan(P.V, esize, sp);
  if (!pass && !walk && !streaming && !make_plan(P.V, esize, extra, topk, topp, pl))
    return SPEC_ERR_UNSUPPORTED;
  // the caller's workspace must hold what the size query promised for the shape
  const bool chain = P.mode == sv::kModeChain;
  const size_t promised =
      layout(P.nseq, n_units, stream_slices(P.V, esize),
             chain ? pass_records(P.nseq, P.gamma, P.V, esize)
                   : walk_records(P.nseq, P.ups, P.V, esize),
             chain ? pass_filter_bytes(P.nseq, P.gamma, P.V, esize) : 0)
          .total;
  if (workspace_bytes < promised) return SPEC_ERR_INVALID_ARG;
  const long long rows = pass   ? static_cast<long long>(P.nseq) * (2 * P.gamma + 1)
                         : walk ? static_cast<long long>(P.nseq) * 2 * P.ups
                                : 0;
  const long long recs = rows * pp.cpr * sv::chain_records_per_chunk();
  const size_t fbytes = pass && topk ? pass_filter_bytes(P.nseq, P.gamma, P.V, esize) : 0;
  const Layout L = layout(P.nseq, n_units, streaming ? sp.slices : 0, recs, fbytes);
  if (workspace_bytes < L.total) return SPEC_ERR_INVALID_ARG;
  char *ws = static_cast<char *>(workspace);
  cudaError_t e = cudaMemsetAsync(ws, 0, L.zero_bytes, stream);
  if (e != cudaSuccess) return map_cuda(e);
  P.counters = reinterpret_cast<uint32_t *>(ws + L.counters);
  P.outs = reinterpret_cast<sv::UnitOut *>(ws + L.outs);
  P.stats = reinterpret_cast<sv::UnitStats *>(ws + L.stats);
  P.final_unit = reinterpret_cast<int32_t *>(ws + L.final_unit);
  P.refine = reinterpret_cast<int4 *>(ws + L.refine);
  P.refine_ctr = reinterpret_cast<uint32_t *>(ws + L.wq_ctr) + 3;
  P.rbar = reinterpret_cast<uint32_t *>(ws + L.wq_ctr) + 4;
  P.rpart = reinterpret_cast<sv::RefinePart *>(ws + L.rpart);
  P.rc = reinterpret_cast<double *>(ws + L.rc);
  P.err = reinterpret_cast<uint32_t *>(ws + L.err);
  P.n_units = static_cast<int>(n_units);
  if (pass) {
    P.ring = pp.ring;
    P.slot_bytes = pp.slot_bytes;
    P.chunk_elems = pp.chunk_elems;
    P.cpr = pp.cpr;
    P.steps = pp.steps;
    P.srec = reinterpret_cast<unsigned long long *>(ws + L.srec);
    P.pseqw = reinterpret_cast<unsigned long long *>(ws + L.pseq);
    P.near_list = reinterpret_cast<int32_t *>(ws + L.near_list);
    P.pctr = reinterpret_cast<uint32_t *>(ws + L.pctr);
    P.nblk = static_cast<int>(pass_blocks(P.V));
    if (topk) {  // block maxima, then 256-byte aligned per-row filter records
      P.bmax = ws + L.bmax;
      P.frec = reinterpret_cast<float2 *>(
          ws + L.bmax + align_up(static_cast<size_t>(rows * P.nblk * esize), 256));
    } else {
      P.bmax = nullptr;
      P.frec = nullptr;
    }
    P.first_wait = g_first_wait.load(std::memory_order_relaxed);
    // rows kernel: its control block, then the ring of chunk slots
    const size_t rows_off = align_up(sv::chain_rows_ctl_bytes(), 128);
    P.data_off = static_cast<int>(rows_off);
    e = sv::launch_chain(P, esize, exp2_table(), rows_off + static_cast<size_t>(pp.ring) * pp.slot_bytes,
                         stream);
  } else if (walk) {
    P.ring = pp.ring;
    P.slot_bytes = pp.slot_bytes;
    P.chunk_elems = pp.chunk_elems;
    P.cpr = pp.cpr;
    P.steps = pp.steps;
    P.srec = reinterpret_cast<unsigned long long *>(ws + L.srec);
    P.bmax = nullptr;
    P.frec = nullptr;
    P.first_wait = g_first_wait.load(std::memory_order_relaxed);
    // the rows kernel skips the draft rows of leaves: first children first
    int32_t *fc = reinterpret_cast<int32_t *>(ws + L.first_child);
    e = sv::launch_first_child(P.parent, P.nseq, P.ups, fc, stream);
    if (e != cudaSuccess) return map_cuda(e);
    P.first_child = fc;
    const size_t rows_off = align_up(sv::chain_rows_ctl_bytes(), 128);
    P.data_off = static_cast<int>(rows_off);
    e = sv::launch_tree_walk(P, esize, rows_off + static_cast<size_t>(pp.ring) * pp.slot_bytes,
                             stream);
  } else if (streaming) {
    P.slice = sp.slice;
    P.cluster = sp.slices;
    P.data_off = static_cast<int>(sp.data_off);
    P.hist_off = 0;
    P.ring = sp.ring;
    P.slot_bytes = sp.slot_bytes;
    P.chunks = sp.chunks;
    P.slice_blocks = sp.chunks * sv::kBlocksPerChunk + 1;
    P.unit_done = reinterpret_cast<uint32_t *>(ws + L.unit_done);
    P.w_done = reinterpret_cast<uint32_t *>(ws + L.w_done);
    P.partials = reinterpret_cast<sv::SlicePartial *>(ws + L.partials);
    P.dstate = reinterpret_cast<sv::DrawState *>(ws + L.dstate);
    P.wpart = reinterpret_cast<float *>(ws + L.wpart);
    P.wblk = reinterpret_cast<float *>(ws + L.wblk);
    P.wq = reinterpret_cast<int4 *>(ws + L.wq);
    P.wq_ctr = reinterpret_cast<uint32_t *>(ws + L.wq_ctr);
    P.wq_cap = static_cast<int>(L.wq_cap);
    // tags this call's queue entries (stale ones never match); one counter for
    // all host threads, never 0
    static std::atomic<uint32_t> epoch{0};
    uint32_t ep = epoch.fetch_add(1u, std::memory_order_relaxed) + 1u;
    if (ep == 0u) ep = epoch.fetch_add(1u, std::memory_order_relaxed) + 1u;
    P.epoch = ep;
    if (P.mode == sv::kModeTree) {
      int32_t *fc = reinterpret_cast<int32_t *>(ws + L.first_child);
      e = sv::launch_first_child(P.parent, P.nseq, P.ups, fc, stream);
      if (e != cudaSuccess) return map_cuda(e);
      P.first_child = fc;
    }
    e = sv::launch_stream(P, esize, sp.smem, stream);
  } else {
    if (n_units * pl.cluster > 0x7FFFFFFFll) return SPEC_ERR_INVALID_ARG;
    P.slice = pl.slice;
    P.cluster = pl.cluster;
    P.data_off = static_cast<int>(pl.data_off);
    P.hist_off = static_cast<int>(pl.hist_off);
    P.mass_off = static_cast<int>(pl.mass_off);
    e = sv::launch_units(P, esize, vec, static_cast<int>(n_units), pl.smem, stream);
  }
  if (e != cudaSuccess) return map_cuda(e);
  if (!pass) {  // the streaming chain path has its own precise redraw; trees take this one
    e = sv::launch_refine(P, esize, exp2_table(), stream);
    if (e != cudaSuccess) return map_cuda(e);
  }
  if (out_residual) {
    e = sv::launch_residual(P, esize, out_residual, stream);
    if (e != cudaSuccess) return map_cuda(e);
  }
  return SPEC_OK;
}

}  // namespace

namespace sv {

// Host-side argument checks of a chain verification call (everything except
// the workspace), shared by spec_verify_chain and spec_verify_chain_static.
// SPEC_OK with B == 0 means there is nothing to do.
spec_status check_chain_args(const void *target_logits, int64_t ld_target,
                             const void *draft_logits, int64_t ld_draft, spec_dtype dtype, int B,
                             int gamma, int V, const int32_t *draft_tokens,
                             spec_policy target_policy, spec_policy draft_policy,
                             const int32_t *out_num_accepted, const int32_t *out_tokens) {
  const int esize = esize_of(dtype);
  if (esize == 0 || B < 0 || gamma < 0 || gamma > kMaxGamma || V < 1) return SPEC_ERR_INVALID_ARG;
  if (B == 0) return SPEC_OK;
  if (!target_logits || ld_target < V || !target_policy.temperature ||
      !draft_policy.temperature || !out_num_accepted || !out_tokens)
    return SPEC_ERR_INVALID_ARG;
  if (gamma > 0 && (!draft_logits || ld_draft < V || !draft_tokens)) return SPEC_ERR_INVALID_ARG;
  return SPEC_OK;
}

}  // namespace sv

extern "C" {

spec_status spec_set_wait_limit(int64_t cycles) {
  g_first_wait.store(cycles < 0 ? sv::kWaitLimitCycles : static_cast<long long>(cycles),
                     std::memory_order_relaxed);
  return SPEC_OK;
}

spec_status spec_set_profile_events(void *start_event, void *stop_event) {
  return sv::set_profile_events(start_event, stop_event) ? SPEC_OK : SPEC_ERR_INVALID_ARG;
}

const char *spec_status_string(spec_status status) {
  switch (status) {
    case SPEC_OK: return "SPEC_OK";
    case SPEC_ERR_INVALID_ARG: return "SPEC_ERR_INVALID_ARG: an argument failed a host-side check";
    case SPEC_ERR_CUDA: return "SPEC_ERR_CUDA: a CUDA launch failed";
    case SPEC_ERR_UNSUPPORTED: return "SPEC_ERR_UNSUPPORTED: shape not supported by this build";
  }
  return "unknown spec_status";
}

size_t spec_verify_chain_workspace_size(int B, int gamma, int V, spec_dtype dtype) {
  const int esize = esize_of(dtype);
  if (B < 0 || gamma < 0 || V < 1 || esize == 0) return 0;
  return layout(B, static_cast<long long>(B) * (gamma + 1), stream_slices(V, esize),
                pass_records(B, gamma, V, esize), pass_filter_bytes(B, gamma, V, esize))
      .total;
}

size_t spec_verify_tree_workspace_size(int T, int N, int V, spec_dtype dtype) {
  const int esize = esize_of(dtype);
  if (T < 0 || N < 0 || V < 1 || esize == 0) return 0;
  return layout(T, static_cast<long long>(T) * N, stream_slices(V, esize),
                walk_records(T, N, V, esize), 0)
      .total;
}

spec_status spec_verify_chain(const void *target_logits, int64_t ld_target,
                              const void *draft_logits, int64_t ld_draft, spec_dtype dtype, int B,
                              int gamma, int V, const int32_t *draft_tokens,
                              spec_policy target_policy, spec_policy draft_policy, uint64_t seed,
                              const float *uniform_override, int32_t *out_num_accepted,
                              int32_t *out_tokens, uint32_t *out_flags, float *out_residual,
                              void *workspace, size_t workspace_bytes, spec_stream_t stream) {
  const spec_status chk = sv::check_chain_args(target_logits, ld_target, draft_logits, ld_draft,
                                               dtype, B, gamma, V, draft_tokens, target_policy,
                                               draft_policy, out_num_accepted, out_tokens);
  if (chk != SPEC_OK || B == 0) return chk;
  if (!workspace) return SPEC_ERR_INVALID_ARG;
  const int esize = esize_of(dtype);
  sv::Params P = {};
  P.target = target_logits;
  P.ld_t = ld_target;
  P.draft = gamma > 0 ? draft_logits : target_logits;
  P.ld_d = gamma > 0 ? ld_draft : ld_target;
  P.V = V;
  P.mode = sv::kModeChain;
  P.nseq = B;
  P.ups = gamma + 1;
  P.gamma = gamma;
  P.max_depth = gamma;
  P.tokens = draft_tokens;
  P.parent = nullptr;
  P.Tp = target_policy.temperature;
  P.Tq = draft_policy.temperature;
  P.kp = target_policy.top_k;
  P.kq = draft_policy.top_k;
  P.pp = target_policy.top_p;
  P.pq = draft_policy.top_p;
  P.mp = target_policy.min_p;
  P.mq = draft_policy.min_p;
  P.seed = seed;
  P.uov = uniform_override;
  P.out_num = out_num_accepted;
  P.out_path = nullptr;
  P.out_tokens = out_tokens;
  P.out_flags = out_flags;
  return run_units(P, esize, static_cast<long long>(B) * (gamma + 1), 0, out_residual, workspace,
                   workspace_bytes, reinterpret_cast<cudaStream_t>(stream), gamma > 0);
}

spec_status spec_verify_tree(const void *target_logits, int64_t ld_target,
                             const void *draft_logits, int64_t ld_draft, spec_dtype dtype, int T,
                             int N, int V, int max_depth, const int32_t *node_tokens,
                             const int32_t *parent, spec_policy target_policy,
                             spec_policy draft_policy, uint64_t seed,
                             const float *uniform_override, int32_t *out_num_accepted,
                             int32_t *out_path, int32_t *out_tokens, uint32_t *out_flags,
                             float *out_residual, void *workspace, size_t workspace_bytes,
                             spec_stream_t stream) {
  const int esize = esize_of(dtype);
  if (esize == 0 || T < 0 || N < 1 || N > kMaxNodes || V < 1 || max_depth < 0)
    return SPEC_ERR_INVALID_ARG;
  if (T == 0) return SPEC_OK;
  if (!target_logits || ld_target < V || !draft_logits || ld_draft < V || !node_tokens ||
      !parent || !target_policy.temperature || !draft_policy.temperature || !out_num_accepted ||
      !out_path || !out_tokens || !workspace)
    return SPEC_ERR_INVALID_ARG;
  sv::Params P = {};
  P.target = target_logits;
  P.ld_t = ld_target;
  P.draft = draft_logits;
  P.ld_d = ld_draft;
  P.V = V;
  P.mode = sv::kModeTree;
  P.nseq = T;
  P.ups = N;
  P.gamma = 0;
  P.max_depth = max_depth;
  P.tokens = node_tokens;
  P.parent = parent;
  P.Tp = target_policy.temperature;
  P.Tq = draft_policy.temperature;
  P.kp = target_policy.top_k;
  P.kq = draft_policy.top_k;
  P.pp = target_policy.top_p;
  P.pq = draft_policy.top_p;
  P.mp = target_policy.min_p;
  P.mq = draft_policy.min_p;
  P.seed = seed;
  P.uov = uniform_override;
  P.out_num = out_num_accepted;
  P.out_path = out_path;
  P.out_tokens = out_tokens;
  P.out_flags = out_flags;
  return run_units(P, esize, static_cast<long long>(T) * N, 2 * sizeof(int) * N, out_residual,
                   workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream), true);
}

spec_status spec_tree_mask(const int32_t *parent, int T, int N, int max_depth, uint64_t *out_mask,
                           int32_t *out_position, uint32_t *out_flags, spec_stream_t stream) {
  if (T < 0 || N < 1 || N > kMaxNodes || max_depth < 0) return SPEC_ERR_INVALID_ARG;
  if (T == 0) return SPEC_OK;
  if (!parent || !out_mask || !out_position) return SPEC_ERR_INVALID_ARG;
  return map_cuda(sv::launch_tree_mask(parent, T, N, max_depth, out_mask, out_position, out_flags,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

spec_status spec_overlap(const void *target_logits, int64_t ld_target, const void *draft_logits,
                         int64_t ld_draft, spec_dtype dtype, int B, int gamma, int V,
                         spec_policy target_policy, spec_policy draft_policy, float *out_beta,
                         uint32_t *out_flags, spec_stream_t stream) {
  const int esize = esize_of(dtype);
  if (esize == 0 || B < 0 || gamma < 0 || gamma > kMaxGamma || V < 1) return SPEC_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * gamma == 0) return SPEC_OK;
  if (!target_logits || !draft_logits || !out_beta || !target_policy.temperature ||
      !draft_policy.temperature || ld_target < V || ld_draft < V)
    return SPEC_ERR_INVALID_ARG;
  if (target_policy.top_k || draft_policy.top_k || target_policy.top_p || draft_policy.top_p ||
      target_policy.min_p || draft_policy.min_p)
    return SPEC_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * gamma > 0x7FFFFFFFll / 8) return SPEC_ERR_INVALID_ARG;  // headroom for clusters
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (out_flags) {
    const cudaError_t e = cudaMemsetAsync(out_flags, 0, static_cast<size_t>(B) * sizeof(uint32_t), st);
    if (e != cudaSuccess) return map_cuda(e);
  }
  return map_cuda(sv::launch_overlap(target_logits, ld_target, draft_logits, ld_draft, esize, B,
                                     gamma, V, target_policy.temperature,
                                     draft_policy.temperature, out_beta, out_flags, st));
}

size_t spec_typical_workspace_size(int B, int gamma, int V, spec_dtype dtype) {
  const int esize = esize_of(dtype);
  if (B < 0 || gamma < 0 || gamma > kMaxGamma || V < 1 || esize == 0) return 0;
  return sv::typical_workspace_bytes(B, gamma, V, esize);
}

spec_status spec_typical_accept(const void *target_logits, int64_t ld_target, spec_dtype dtype,
                                int B, int gamma, int V, spec_policy target_policy,
                                const int32_t *draft_tokens, float epsilon, float delta,
                                int32_t *out_num_accepted, int32_t *out_tokens,
                                uint32_t *out_flags, void *workspace, size_t workspace_bytes,
                                spec_stream_t stream) {
  const int esize = esize_of(dtype);
  if (esize == 0 || B < 0 || gamma < 0 || gamma > kMaxGamma || V < 1) return SPEC_ERR_INVALID_ARG;
  if (!(epsilon >= 0.f) || !(delta >= 0.f) || epsilon == INFINITY || delta == INFINITY)
    return SPEC_ERR_INVALID_ARG;
  if (B == 0) return SPEC_OK;
  if (!target_logits || !target_policy.temperature || (gamma > 0 && !draft_tokens) ||
      !out_num_accepted || !out_tokens || !workspace || ld_target < V)
    return SPEC_ERR_INVALID_ARG;
  if (target_policy.top_k || target_policy.top_p || target_policy.min_p) return SPEC_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * (gamma + 1) > 0x7FFFFFFFll / 8) return SPEC_ERR_INVALID_ARG;
  if (workspace_bytes < sv::typical_workspace_bytes(B, gamma, V, esize) ||
      (reinterpret_cast<uintptr_t>(workspace) & 7u) != 0)
    return SPEC_ERR_INVALID_ARG;
  return map_cuda(sv::launch_typical(target_logits, ld_target, esize, B, gamma, V,
                                     target_policy.temperature, draft_tokens, epsilon, delta,
                                     out_num_accepted, out_tokens, out_flags, workspace,
                                     reinterpret_cast<cudaStream_t>(stream)));
}

spec_status spec_tree_rerank(const int32_t *parent, const float *confidence, int T, int N, int m,
                             int32_t *out_nodes, int32_t *out_parent, float *out_value,
                             int32_t *out_count, uint32_t *out_flags, spec_stream_t stream) {
  if (T < 0 || N < 1 || N > kMaxNodes || m < 1) return SPEC_ERR_INVALID_ARG;
  if (T == 0) return SPEC_OK;
  if (!parent || !confidence || !out_nodes || !out_parent || !out_count)
    return SPEC_ERR_INVALID_ARG;
  return map_cuda(sv::launch_tree_rerank(parent, confidence, T, N, m, out_nodes, out_parent,
                                         out_value, out_count, out_flags,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
