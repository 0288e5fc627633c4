// Chain verification in one streaming pass (rows 16-byte aligned, no top-k,
// gamma <= 31).
//
// Every logit row of the batch - the gamma + 1 target rows and gamma draft
// rows of each sequence - is cut into chunks of 32 KB.  Chunks are numbered
// sequence-major and handed out round-robin (CTA b takes chunks b, b + grid,
// ...), so the whole grid sweeps the batch front to back and sequences
// complete one after another.  Each CTA has three roles:
//
//   warp 8 (producer): streams the CTA's chunks into a ring of shared-memory
//     slots with bulk asynchronous copies (cp.async.bulk, one "full" and one
//     "empty" mbarrier per slot), with each chunk's description beside it.
//     When the consumers hand a slot back it refills it;
//   warps 0-7 (consumers): each reduces its eighth of the chunk to one 64-bit
//     record, the (max, sum of 2^((z - max) log2(e) / T)) of a sampling row or
//     the (finite max, lowest index + 1) of a greedy row, and stores it in one
//     access (a record is never seen half written; zero means not written);
//     the last warp done with a chunk adds it to its sequence's counter (a
//     relaxed add, no fence: only a hint);
//   warps 9-12 (the draw group): a small scheduler that takes, in order of
//     priority, (1) the search of its owned sequence once the sequence's
//     weight jobs are all counted, (2) the decision of its next owned sequence
//     (b, b + grid, ...) once the sequence's chunk counter is complete, (3)
//     its next weight job once that job's draw descriptor is published, and
//     (4) precise-redraw jobs once it has nothing else left.  All of this is
//     described with the distributed draws below.
//
// A decision merges the records (retrying while any still reads zero) into
// each row's softmax normaliser (or argmax), runs the acceptance tests of all
// gamma positions at once (one lane each: u < min(1, p/q) with Philox
// uniforms, or the greedy rule), finds the first rejection j with a warp
// ballot and publishes the draw at j: the correction from [p_j - q_j]_+ or the
// bonus from p_gamma.  The draw's two rows, streamed a few microseconds
// earlier, are re-read from L2 by weight jobs spread over many CTAs.
//
// No fence sits on the streaming path or on the draw path: records, draw
// descriptors and step totals are 64-bit entries that validate themselves
// (zero means not yet written), and counters are relaxed hints.  The draw
// groups wait on other CTAs' progress, so the grid is launched cooperatively
// (all CTAs resident, two per SM); every wait is bounded.
//
// Exponent arithmetic: 2^((z - m) k) with z - m computed exactly (one
// rounding in the product), in the records, the merge, the acceptance test
// and the draw alike, so the normalisers and the draw weights share their
// scale.
#include <mutex>

#include "ops.cuh"
#include "precise_row.cuh"

namespace sv {

constexpr int kPConsumerWarps = 8;
constexpr int kPProducerWarp = 8;
constexpr int kPDrawWarp0 = 9;
constexpr int kPDrawWarps = 4;
constexpr int kPThreads = (kPConsumerWarps + 1 + kPDrawWarps) * 32;  // 416
constexpr int kPDrawThreads = kPDrawWarps * 32;
constexpr int kPMaxRing = 8;
constexpr int kPMaxGamma = 31;
constexpr int kPMaxRows = 2 * kPMaxGamma + 1;
constexpr int kPStep = 256;                        // entries per draw-search step
constexpr int kPWeightJobs = 16;                   // weight jobs per draw (at most)
static_assert(kPWeightJobs <= 32, "a group's weight-job residues are sorted by one warp");
constexpr int kPPreciseJobs = kPassPreciseJobs;    // precise jobs per phase (at most)
constexpr long long kPPollLimitNs = 2000000000ll;  // give up waiting after about 2 s
constexpr uint32_t kNoIndex = 0x3FFFFFFFu;         // record index: no finite entry
constexpr uint32_t kBadBit = 0x80000000u;          // record index bit: NaN or +inf seen

// What the producer tells the consumers about the chunk in a slot.
struct SlotInfo {
  const void *gl;  // the chunk in global memory
  long long rec;   // index of the chunk's first record
  int n;           // entries
  int nb;          // entries copied to shared memory
  float k;         // log2(e) / T, 0 for a greedy row
  int arg;         // greedy row: argmax record
  int v0;          // vocabulary index of the chunk's first entry
  int seq;         // sequence of the chunk
};

struct PassRow {
  float m, S;  // merged max and sum (sampling rows) or argmax value (greedy rows)
  int a;       // argmax index (greedy rows; fallback rows)
  int bad;     // NaN / +inf seen, or nothing finite
};

struct PassCtl {
  unsigned long long full[kPMaxRing];
  unsigned long long empty[kPMaxRing];
  SlotInfo info[kPMaxRing];
  int slot_done[kPMaxRing];  // consumer warps finished with the slot's chunk
  PassRow row[kPMaxRows];
  RowDesc desc[kPMaxRows];
  double W;
  double t_rel;
  int step;
  int j;
  uint32_t flags;
  int pos_flags[kPMaxGamma + 1];
  int redo;
  int red_i[kPDrawWarps];
  float red_v[kPDrawWarps];
  // job scheduling
  PassSeq ps;
  double pred[2][kPDrawWarps];
  float tab_hi[64], tab_lo[64];
  long long idle_t0;
  int act, next_dec, next_f, next_k, job_v, job_s;
  int tokx[kPMaxGamma + 1];
  float u_draw;  // the draw uniform at the decided position
  int fj_s[32], fj_k[32];  // the group's weight-job residues, ascending
  int fj_i, fj_m;
  int next_srch;   // owned sequence whose weight jobs are awaited (-1: none)
  int held_v;      // claimed precise job id not yet run (-1: none)
  PassSeq ps_own;  // its descriptor
};

__device__ __forceinline__ void draw_sync() {
  asm volatile("bar.sync 2, 128;" ::: "memory");
}

__device__ __forceinline__ long long pass_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return static_cast<long long>(t);
}

__device__ __forceinline__ uint32_t ld_volatile_pass(const uint32_t *p) {
  return *reinterpret_cast<const volatile uint32_t *>(p);
}

__device__ __forceinline__ void mbar_arrive1(unsigned long long *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// 2^((z - m) k): the exponent form every step of this kernel uses.
__device__ __forceinline__ float pexp(float z, float m, float k) {
  return fast_exp2(__fmul_rn(__fsub_rn(z, m), k));
}

// Probability of entry v with logit z under a row descriptor.
__device__ __forceinline__ float pprob(const RowDesc &d, float z, int v) {
  if (d.onehot) return v == d.a ? 1.f : 0.f;
  return pexp(z, d.m, d.k) * d.invS;
}

// Where work item k (a chunk) lives.
struct ChunkInfo {
  int seq, r, c, n;  // sequence, row within the sequence, chunk, entries
  long long row;     // global row (target rows first: r <= gamma)
  bool draft;
};

__device__ __forceinline__ ChunkInfo chunk_info(const Params &P, long long k) {
  ChunkInfo ci;
  const int rps = 2 * P.gamma + 1;
  const int per_seq = rps * P.cpr;
  const int k32 = static_cast<int>(k);  // the host keeps the chunk count below 2^31
  ci.seq = k32 / per_seq;
  const int rem = k32 - ci.seq * per_seq;
  ci.r = rem / P.cpr;
  ci.c = rem - ci.r * P.cpr;
  ci.n = min(P.chunk_elems, P.V - ci.c * P.chunk_elems);
  ci.draft = ci.r > P.gamma;
  ci.row = ci.draft ? static_cast<long long>(ci.seq) * P.gamma + (ci.r - P.gamma - 1)
                    : static_cast<long long>(ci.seq) * (P.gamma + 1) + ci.r;
  return ci;
}

// Policy of a row: greedy (argmax) or sampling with k = log2(e) / T.
__device__ __forceinline__ bool row_is_arg(float T) { return !(T > 0.f) || T == INFINITY; }

// ---------------------------------------------------------------------------
// consumers: one record per warp per chunk
// ---------------------------------------------------------------------------

template <typename TE>
__device__ __forceinline__ void load_vec(const TE *s, float z[8]);
template <>
__device__ __forceinline__ void load_vec<uint16_t>(const uint16_t *s, float z[8]) {
  const uint4 w = *reinterpret_cast<const uint4 *>(s);
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    z[2 * i] = __uint_as_float(ws[i] << 16);
    z[2 * i + 1] = __uint_as_float(ws[i] & 0xFFFF0000u);
  }
}
template <>
__device__ __forceinline__ void load_vec<float>(const float *s, float z[8]) {
  const float4 a = *reinterpret_cast<const float4 *>(s);
  const float4 b = *reinterpret_cast<const float4 *>(s + 4);
  z[0] = a.x; z[1] = a.y; z[2] = a.z; z[3] = a.w;
  z[4] = b.x; z[5] = b.y; z[6] = b.z; z[7] = b.w;
}

// Record of this warp's part [e0, e1) of a chunk: entries below nb come from
// shared memory (groups of 8), the rest (fewer than 8) from global memory.
template <typename TE>
__device__ float2 chunk_record(const TE *sm, const TE *gl, int e0, int e1, int nb, int v0,
                               bool arg, float k) {
  const int lane = threadIdx.x & 31;
  if (arg) {
    float bv = -INFINITY;
    uint32_t bi = kNoIndex, bad = 0u;
    for (int base = e0 + lane * 8; base < e1; base += 256) {
      float z[8];
      if (base + 8 <= nb) {
        load_vec<TE>(sm + base, z);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) z[e] = base + e < e1 ? to_f32(gl[base + e]) : -INFINITY;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float x = z[e];
        if (x != x || x == INFINITY) {
          if (base + e < e1) bad = 1u;
        } else if (x > bv) {
          bv = x;
          bi = static_cast<uint32_t>(v0 + base + e);
        }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float v2 = __shfl_xor_sync(0xFFFFFFFFu, bv, off);
      const uint32_t i2 = __shfl_xor_sync(0xFFFFFFFFu, bi, off);
      bad |= __shfl_xor_sync(0xFFFFFFFFu, bad, off);
      if (v2 > bv || (v2 == bv && i2 < bi)) {
        bv = v2;
        bi = i2;
      }
    }
    return make_float2(bv, __uint_as_float((bi + 1u) | (bad ? kBadBit : 0u)));
  }
  // sampling row: one pass with a running max; the packed partial sums are
  // rescaled (folded into S) whenever the max grows
  float m = -INFINITY, S = 0.f;
  bool nan = false;
  const uint64_t k2 = pack2(k, k);
  uint64_t acc0 = 0ull, acc1 = 0ull;
  for (int base = e0 + lane * 8; base < e1; base += 256) {
    float z[8];
    if (base + 8 <= nb) {
      load_vec<TE>(sm + base, z);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) z[e] = base + e < e1 ? to_f32(gl[base + e]) : -INFINITY;
    }
    const float gm = fmaxf(fmaxf(fmaxf(z[0], z[1]), fmaxf(z[2], z[3])),
                           fmaxf(fmaxf(z[4], z[5]), fmaxf(z[6], z[7])));
    if (gm > m) {
      if (m > -INFINITY) {
        const float sc = fast_exp2(__fmul_rn(__fsub_rn(m, gm), k));
        S = (S + hsum2(fadd2(acc0, acc1))) * sc;
      }
      acc0 = acc1 = 0ull;
      m = gm;
    }
    if (m == -INFINITY) {
#pragma unroll
      for (int e = 0; e < 8; ++e) nan |= z[e] != z[e];
      continue;
    }
    const uint64_t nm2 = pack2(-m, -m);
    acc0 = fadd2(acc0, ex2_pair(fmul2(fadd2(pack2(z[0], z[1]), nm2), k2)));
    acc1 = fadd2(acc1, ex2_pair(fmul2(fadd2(pack2(z[2], z[3]), nm2), k2)));
    acc0 = fadd2(acc0, ex2_pair(fmul2(fadd2(pack2(z[4], z[5]), nm2), k2)));
    acc1 = fadd2(acc1, ex2_pair(fmul2(fadd2(pack2(z[6], z[7]), nm2), k2)));
  }
  S += hsum2(fadd2(acc0, acc1));
  if (nan) S = __int_as_float(0x7FC00000);  // NaN marks the record bad
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, off);
    const float S2 = __shfl_xor_sync(0xFFFFFFFFu, S, off);
    if (S2 != S2 || S != S) {
      S = __int_as_float(0x7FC00000);
      m = fmaxf(m, m2);
    } else if (m2 > -INFINITY) {
      if (m == -INFINITY) {
        m = m2;
        S = S2;
      } else {
        const float M = fmaxf(m, m2);
        S = S * fast_exp2(__fmul_rn(__fsub_rn(m, M), k)) +
            S2 * fast_exp2(__fmul_rn(__fsub_rn(m2, M), k));
        m = M;
      }
    }
  }
  return make_float2(m, S);
}

// Warp merge of per-lane (max, sum) pairs; a NaN sum marks the record bad.
__device__ __forceinline__ float2 warp_merge_ms(float m, float S, float k) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, off);
    const float S2 = __shfl_xor_sync(0xFFFFFFFFu, S, off);
    if (S2 != S2 || S != S) {
      S = __int_as_float(0x7FC00000);
      m = fmaxf(m, m2);
    } else if (m2 > -INFINITY) {
      if (m == -INFINITY) {
        m = m2;
        S = S2;
      } else {
        const float M = fmaxf(m, m2);
        S = S * fast_exp2(__fmul_rn(__fsub_rn(m, M), k)) +
            S2 * fast_exp2(__fmul_rn(__fsub_rn(m2, M), k));
        m = M;
      }
    }
  }
  return make_float2(m, S);
}

// Sampling-row record when every group of 8 entries of the warp's part is in
// shared memory: each lane loads all of its groups, takes one max and one sum
// of 2^((z - max) k) over independent packed chains.
template <typename TE>
__device__ float2 sample_record_fast(const TE *sm, int e0, int e1, float k);

template <>
__device__ float2 sample_record_fast<uint16_t>(const uint16_t *sm, int e0, int e1, float k) {
  const int lane = threadIdx.x & 31;
  constexpr int G = 8;  // 2048 entries per warp
  uint4 w[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const int base = e0 + g * 256 + lane * 8;
    w[g] = base < e1 ? *reinterpret_cast<const uint4 *>(sm + base)
                     : make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
  }
  uint32_t h[G];
#pragma unroll
  for (int g = 0; g < G; ++g) h[g] = bf16x2_max(bf16x2_max(w[g].x, w[g].y), bf16x2_max(w[g].z, w[g].w));
  const uint32_t hh = bf16x2_max(bf16x2_max(bf16x2_max(h[0], h[1]), bf16x2_max(h[2], h[3])),
                                 bf16x2_max(bf16x2_max(h[4], h[5]), bf16x2_max(h[6], h[7])));
  const float m = fmaxf(__uint_as_float(hh << 16), __uint_as_float(hh & 0xFFFF0000u));
  float S = 0.f;
  if (m == -INFINITY) {  // nothing but -inf and NaN: look for NaN
    bool nan = false;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const uint32_t ws[4] = {w[g].x, w[g].y, w[g].z, w[g].w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
        nan |= (ws[i] & 0x7FFFu) > 0x7F80u || (ws[i] & 0x7FFF0000u) > 0x7F800000u;
    }
    if (nan) S = __int_as_float(0x7FC00000);
  } else {
    const uint64_t nm2 = pack2(-m, -m), k2 = pack2(k, k);
    // eight independent chains (two per word slot, alternating groups)
    uint64_t a[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) a[c] = 0ull;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const int o = (g & 1) * 4;
      a[o + 0] = fadd2(a[o + 0], ex2_pair(fmul2(fadd2(bf16x2_to_pair(w[g].x), nm2), k2)));
      a[o + 1] = fadd2(a[o + 1], ex2_pair(fmul2(fadd2(bf16x2_to_pair(w[g].y), nm2), k2)));
      a[o + 2] = fadd2(a[o + 2], ex2_pair(fmul2(fadd2(bf16x2_to_pair(w[g].z), nm2), k2)));
      a[o + 3] = fadd2(a[o + 3], ex2_pair(fmul2(fadd2(bf16x2_to_pair(w[g].w), nm2), k2)));
    }
    S = hsum2(fadd2(fadd2(fadd2(a[0], a[1]), fadd2(a[2], a[3])),
                    fadd2(fadd2(a[4], a[5]), fadd2(a[6], a[7]))));
  }
  return warp_merge_ms(m, S, k);
}

template <>
__device__ float2 sample_record_fast<float>(const float *sm, int e0, int e1, float k) {
  const int lane = threadIdx.x & 31;
  constexpr int G = 4;  // 1024 entries per warp
  float4 a[G], b[G];
  const float4 ninf = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const int base = e0 + g * 256 + lane * 8;
    a[g] = base < e1 ? *reinterpret_cast<const float4 *>(sm + base) : ninf;
    b[g] = base < e1 ? *reinterpret_cast<const float4 *>(sm + base + 4) : ninf;
  }
  float mg[G];
#pragma unroll
  for (int g = 0; g < G; ++g)
    mg[g] = fmaxf(fmaxf(fmaxf(a[g].x, a[g].y), fmaxf(a[g].z, a[g].w)),
                  fmaxf(fmaxf(b[g].x, b[g].y), fmaxf(b[g].z, b[g].w)));
  const float m = fmaxf(fmaxf(mg[0], mg[1]), fmaxf(mg[2], mg[3]));
  float S = 0.f;
  if (m == -INFINITY) {
    bool nan = false;
#pragma unroll
    for (int g = 0; g < G; ++g)
      nan |= a[g].x != a[g].x || a[g].y != a[g].y || a[g].z != a[g].z || a[g].w != a[g].w ||
             b[g].x != b[g].x || b[g].y != b[g].y || b[g].z != b[g].z || b[g].w != b[g].w;
    if (nan) S = __int_as_float(0x7FC00000);
  } else {
    const uint64_t nm2 = pack2(-m, -m), k2 = pack2(k, k);
    uint64_t s0 = 0ull, s1 = 0ull, s2 = 0ull, s3 = 0ull;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      s0 = fadd2(s0, ex2_pair(fmul2(fadd2(pack2(a[g].x, a[g].y), nm2), k2)));
      s1 = fadd2(s1, ex2_pair(fmul2(fadd2(pack2(a[g].z, a[g].w), nm2), k2)));
      s2 = fadd2(s2, ex2_pair(fmul2(fadd2(pack2(b[g].x, b[g].y), nm2), k2)));
      s3 = fadd2(s3, ex2_pair(fmul2(fadd2(pack2(b[g].z, b[g].w), nm2), k2)));
    }
    S = hsum2(fadd2(fadd2(s0, s1), fadd2(s2, s3)));
  }
  return warp_merge_ms(m, S, k);
}

template <typename TE>
__device__ void consumer_loop(const Params &P, PassCtl &ctl, unsigned char *ring,
                              long long total) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NS = P.ring;
  const int EW = P.chunk_elems / kPConsumerWarps;  // entries per warp (a multiple of 256)
  int i = 0;
  for (long long k = blockIdx.x; k < total; k += gridDim.x, ++i) {
    const int slot = i % NS;
    const uint32_t phase = static_cast<uint32_t>(i / NS) & 1u;
    if (!mbar_wait_bounded(&ctl.full[slot], phase)) {
      if (lane == 0) atomicOr(P.err, 1u);
      mbar_wait_bounded(&ctl.full[slot], phase);  // do not leave a copy in flight
    }
    const SlotInfo si = ctl.info[slot];
    const TE *sm = reinterpret_cast<const TE *>(ring + static_cast<size_t>(slot) * P.slot_bytes);
    const int e0 = min(si.n, warp * EW), e1 = min(si.n, e0 + EW);
    const float2 rec = (!si.arg && si.nb == si.n && (si.n & 7) == 0)
                           ? sample_record_fast<TE>(sm, e0, e1, si.k)
                           : chunk_record<TE>(sm, static_cast<const TE *>(si.gl), e0, e1, si.nb,
                                              si.v0, si.arg != 0, si.k);
    if (lane == 0) {
      const unsigned long long bits =
          static_cast<unsigned long long>(__float_as_uint(rec.x)) |
          (static_cast<unsigned long long>(__float_as_uint(rec.y)) << 32);
      P.srec[si.rec + warp] = bits;  // one 64-bit store
      // the last warp done with the chunk counts it for its sequence (relaxed,
      // no fence: the records validate themselves, the count only says when
      // to look); it resets the slot's tally before handing the slot back
      if (atomicAdd(&ctl.slot_done[slot], 1) == kPConsumerWarps - 1) {
        ctl.slot_done[slot] = 0;
        asm volatile("red.relaxed.gpu.global.add.u32 [%0], 1;" ::"l"(P.seq_cnt + si.seq) : "memory");
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive1(&ctl.empty[slot]);
  }
}

// ---------------------------------------------------------------------------
// producer: bulk copies into the ring, chunk completion to the counters
// ---------------------------------------------------------------------------

template <typename TE>
__device__ void producer_loop(const Params &P, PassCtl &ctl, unsigned char *ring,
                              long long total) {
  const int NS = P.ring;
  const int CE = P.chunk_elems;
  const long long G = gridDim.x;
  // the consumers of the id-th chunk handed its slot back: its records are stored
  auto wait_done = [&](int id) {
    const int slot = id % NS;
    const uint32_t phase = static_cast<uint32_t>(id / NS) & 1u;
    if (!mbar_wait_bounded(&ctl.empty[slot], phase)) atomicOr(P.err, 1u);
  };
  int i = 0;
  for (long long k = blockIdx.x; k < total; k += G, ++i) {
    const int slot = i % NS;
    if (i >= NS) wait_done(i - NS);
    const ChunkInfo ci = chunk_info(P, k);
    const float T = __ldg((ci.draft ? P.Tq : P.Tp) + ci.seq);
    const bool arg = row_is_arg(T);
    const TE *gl = static_cast<const TE *>(row_ptr(ci.draft ? P.draft : P.target, ci.row,
                                                   ci.draft ? P.ld_d : P.ld_t, sizeof(TE))) +
                   static_cast<long long>(ci.c) * CE;
    const uint32_t bytes = static_cast<uint32_t>(ci.n * sizeof(TE)) / 16u * 16u;
    SlotInfo &si = ctl.info[slot];
    si.gl = gl;
    si.rec = ((static_cast<long long>(ci.seq) * (2 * P.gamma + 1) + ci.r) * P.cpr + ci.c) *
             kPConsumerWarps;
    si.n = ci.n;
    si.nb = static_cast<int>(bytes / sizeof(TE));
    si.k = arg ? 0.f : kLog2e / T;
    si.arg = arg ? 1 : 0;
    si.v0 = ci.c * CE;
    si.seq = ci.seq;
    mbar_arrive_expect_tx(&ctl.full[slot], bytes);
    if (bytes) bulk_g2s_plain(ring + static_cast<size_t>(slot) * P.slot_bytes, gl, bytes,
                              &ctl.full[slot]);
  }
  const int issued = i;
  for (int d = max(0, issued - NS); d < issued; ++d) wait_done(d);
}

// ---------------------------------------------------------------------------
// decide / draw group
// ---------------------------------------------------------------------------

// Merge the records of all 2 gamma + 1 rows of a sequence (draw group):
// row r goes to tpr consecutive threads of one warp (tpr a power of two,
// tpr (2 gamma + 1) <= 128), each loading its records eight at a time
// before merging them.  Returns false (in every thread) while a record still
// reads zero (not yet stored).
__device__ bool merge_rows(const Params &P, PassCtl &ctl, int seq, bool p_arg, bool q_arg,
                           float kp, float kq) {
  const int t = threadIdx.x - kPDrawWarp0 * 32, w = t >> 5;
  const int gamma = P.gamma, rps = 2 * gamma + 1;
  const int R = P.cpr * kPConsumerWarps;
  int tpr = 32;
  while (tpr * rps > kPDrawThreads) tpr >>= 1;
  const int r = t / tpr, sub = t - r * tpr;
  const bool active = r < rps;
  const bool draft = r > gamma;
  const bool arg = draft ? q_arg : p_arg;
  const float k = draft ? kq : kp;
  bool missing = false;
  float m = -INFINITY, S = 0.f;
  int bad = 0;
  float bv = -INFINITY;
  uint32_t bi = kNoIndex;
  if (active) {
    const unsigned long long *rec =
        P.srec + (static_cast<long long>(seq) * rps + r) * static_cast<long long>(R);
    for (int x0 = sub; x0 < R; x0 += 8 * tpr) {
      unsigned long long b[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int x = x0 + i * tpr;
        b[i] = x < R ? __ldcg(rec + x) : 0ull;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (x0 + i * tpr >= R) continue;
        missing |= b[i] == 0ull;
        const float qx = __uint_as_float(static_cast<uint32_t>(b[i]));
        const uint32_t qy = static_cast<uint32_t>(b[i] >> 32);
        if (arg) {
          bad |= static_cast<int>(qy >> 31);
          const uint32_t idx = (qy & ~kBadBit) - 1u;
          if (qx > bv || (qx == bv && idx < bi)) {
            bv = qx;
            bi = idx;
          }
        } else {
          const float qs = __uint_as_float(qy);
          if (qs != qs || qx == INFINITY) bad = 1;
          else online_merge(m, S, qx, qs, k);
        }
      }
    }
  }
  // reduce over the row's tpr threads (every lane of the warp shuffles)
  for (int off = tpr >> 1; off > 0; off >>= 1) {
    const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, off);
    const float S2 = __shfl_xor_sync(0xFFFFFFFFu, S, off);
    const float v2 = __shfl_xor_sync(0xFFFFFFFFu, bv, off);
    const uint32_t i2 = __shfl_xor_sync(0xFFFFFFFFu, bi, off);
    bad |= __shfl_xor_sync(0xFFFFFFFFu, bad, off);
    if (!arg) online_merge(m, S, m2, S2, k);
    if (v2 > bv || (v2 == bv && i2 < bi)) {
      bv = v2;
      bi = i2;
    }
  }
  if (active && sub == 0) {
    PassRow pr;
    if (arg) {
      pr.m = bv;
      pr.S = 0.f;
      pr.a = bi == kNoIndex ? 0 : static_cast<int>(bi);
      pr.bad = (bad || bi == kNoIndex) ? 1 : 0;
    } else {
      pr.m = m;
      pr.S = S;
      pr.a = 0;
      pr.bad = (bad || !(m > -INFINITY) || !(S > 0.f) || S == INFINITY) ? 1 : 0;
    }
    ctl.row[r] = pr;
  }
  const bool any_missing = __any_sync(0xFFFFFFFFu, missing);
  if ((t & 31) == 0) ctl.red_i[w] = any_missing ? 0 : 1;
  draw_sync();
  bool all = true;
  for (int x = 0; x < kPDrawWarps; ++x) all &= ctl.red_i[x] != 0;
  draw_sync();
  return all;
}

// Finite argmax of a whole row (draw group; rows whose sampling statistics
// were not finite).
template <typename TE>
__device__ int finite_argmax_row(const TE *g, int V, PassCtl &ctl) {
  const int t = threadIdx.x - kPDrawWarp0 * 32, lane = t & 31, w = t >> 5;
  float bv = -INFINITY;
  int bi = INT_MAX;
  for (int v = t; v < V; v += kPDrawThreads) {
    const float x = to_f32(g[v]);
    if (x == x && x != INFINITY && x > bv) {
      bv = x;
      bi = v;
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float v2 = __shfl_xor_sync(0xFFFFFFFFu, bv, off);
    const int i2 = __shfl_xor_sync(0xFFFFFFFFu, bi, off);
    argmax_merge(bv, bi, v2, i2);
  }
  if (lane == 0) {
    ctl.red_v[w] = bv;
    ctl.red_i[w] = bi;
  }
  draw_sync();
  float v = -INFINITY;
  int i = INT_MAX;
  for (int x = 0; x < kPDrawWarps; ++x) argmax_merge(v, i, ctl.red_v[x], ctl.red_i[x]);
  draw_sync();
  return i == INT_MAX ? 0 : i;
}

// Eight consecutive logits held as loaded (16 or 32 bytes), converted on use.
template <typename TE>
struct Raw8;
template <>
struct Raw8<uint16_t> {
  uint4 w = make_uint4(0u, 0u, 0u, 0u);
  __device__ __forceinline__ void load(const uint16_t *s) {
    w = *reinterpret_cast<const uint4 *>(s);
  }
  __device__ __forceinline__ void get(float z[8]) const {
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      z[2 * i] = __uint_as_float(ws[i] << 16);
      z[2 * i + 1] = __uint_as_float(ws[i] & 0xFFFF0000u);
    }
  }
};
template <>
struct Raw8<float> {
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = make_float4(0.f, 0.f, 0.f, 0.f);
  __device__ __forceinline__ void load(const float *s) {
    a = *reinterpret_cast<const float4 *>(s);
    b = *reinterpret_cast<const float4 *>(s + 4);
  }
  __device__ __forceinline__ void get(float z[8]) const {
    z[0] = a.x; z[1] = a.y; z[2] = a.z; z[3] = a.w;
    z[4] = b.x; z[5] = b.y; z[6] = b.z; z[7] = b.w;
  }
};

// Draw weights of the 8 entries from `base` given their logits.  Sampling
// rows use packed pairs, rounding exactly like pprob().
__device__ __forceinline__ void weights8(const RowDesc &dp, const RowDesc &dq, int residual,
                                         int base, const float zp[8], const float zq[8],
                                         float w[8]) {
  if (!dp.onehot && (!residual || !dq.onehot)) {
    const uint64_t np2 = pack2(-dp.m, -dp.m), kp2 = pack2(dp.k, dp.k),
                   ip2 = pack2(dp.invS, dp.invS);
    const uint64_t nq2 = pack2(-dq.m, -dq.m), kq2 = pack2(dq.k, dq.k),
                   iq2 = pack2(dq.invS, dq.invS);
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      const uint64_t p2 = fmul2(ex2_pair(fmul2(fadd2(pack2(zp[e], zp[e + 1]), np2), kp2)), ip2);
      if (residual) {
        const uint64_t q2 =
            fmul2(ex2_pair(fmul2(fadd2(pack2(zq[e], zq[e + 1]), nq2), kq2)), iq2);
        float d0, d1;
        unpack2(fadd2(p2, q2 ^ 0x8000000080000000ull), d0, d1);
        w[e] = fmaxf(d0, 0.f);
        w[e + 1] = fmaxf(d1, 0.f);
      } else {
        unpack2(p2, w[e], w[e + 1]);
      }
    }
    return;
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    float x = pprob(dp, zp[e], base + e);
    if (residual) x = fmaxf(x - pprob(dq, zq[e], base + e), 0.f);
    w[e] = x;
  }
}

// Draw weights of 8 entries from `base` (entries at or past V are 0).
template <typename TE>
__device__ __forceinline__ void step_weights(const TE *gp, const TE *gq, const RowDesc &dp,
                                             const RowDesc &dq, int residual, int base, int V,
                                             float w[8]) {
  float zp[8], zq[8];
  const bool full = base + 8 <= V;
  if (full && !dp.onehot) {
    load_vec<TE>(gp + base, zp);
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) zp[e] = (!dp.onehot && base + e < V) ? to_f32(gp[base + e]) : 0.f;
  }
  if (residual) {
    if (full && !dq.onehot) {
      load_vec<TE>(gq + base, zq);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e)
        zq[e] = (!dq.onehot && base + e < V) ? to_f32(gq[base + e]) : 0.f;
    }
  }
  if (!residual) {
#pragma unroll
    for (int e = 0; e < 8; ++e) zq[e] = 0.f;
  }
  weights8(dp, dq, residual, base, zp, zq, w);  // the same arithmetic as the pass
#pragma unroll
  for (int e = 0; e < 8; ++e)
    if (base + e >= V) w[e] = 0.f;
}

// Inverse-CDF draw of the sequence's final token (the whole draw group).
// Returns the token; `margin` is its distance from the nearer boundary.
template <typename TE>
__device__ int pass_draw(const Params &P, PassCtl &ctl, float *step_tot, const TE *gp,
                         const TE *gq, const RowDesc &dp, const RowDesc &dq, int residual,
                         float u, float &margin, double &Wout) {
  const int t = threadIdx.x - kPDrawWarp0 * 32, lane = t & 31, w = t >> 5;
  const int V = P.V, nsteps = P.steps;
  // pass: step totals.  Full steps go four per warp at a time, their loads
  // issued before any of them is used; the ragged last step goes alone.
  constexpr int kU = 4;
  const int nfull = V / kPStep;
  int st0 = w;
  for (; st0 + (kU - 1) * kPDrawWarps < nfull; st0 += kPDrawWarps * kU) {
    Raw8<TE> rp[kU], rq[kU];
#pragma unroll
    for (int q = 0; q < kU; ++q) {
      const int base = (st0 + q * kPDrawWarps) * kPStep + lane * 8;
      if (!dp.onehot) rp[q].load(gp + base);
      if (residual && !dq.onehot) rq[q].load(gq + base);
    }
#pragma unroll
    for (int q = 0; q < kU; ++q) {
      const int base = (st0 + q * kPDrawWarps) * kPStep + lane * 8;
      float zp[8], zq[8], x[8];
      rp[q].get(zp);
      rq[q].get(zq);
      weights8(dp, dq, residual, base, zp, zq, x);
      float s = ((x[0] + x[1]) + (x[2] + x[3])) + ((x[4] + x[5]) + (x[6] + x[7]));
      s = warp_sum(s);
      if (lane == 0) step_tot[st0 + q * kPDrawWarps] = s;
    }
  }
  for (int st = st0; st < nsteps; st += kPDrawWarps) {
    float x[8];
    step_weights<TE>(gp, gq, dp, dq, residual, st * kPStep + lane * 8, V, x);
    float s = ((x[0] + x[1]) + (x[2] + x[3])) + ((x[4] + x[5]) + (x[6] + x[7]));
    s = warp_sum(s);
    if (lane == 0) step_tot[st] = s;
  }
  draw_sync();
  if (w == 0) {
    // total and the owning step: lanes own contiguous runs of steps
    const int per = (nsteps + 31) / 32;
    const int s0 = min(nsteps, lane * per), s1 = min(nsteps, s0 + per);
    double seg = 0.0;
    int lastpos = -1;
    for (int st = s0; st < s1; ++st) {
      seg += static_cast<double>(step_tot[st]);
      if (step_tot[st] > 0.f) lastpos = st;
    }
    double incl = seg;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const double y = __shfl_up_sync(0xFFFFFFFFu, incl, off);
      if (lane >= off) incl += y;
    }
    const double W = __shfl_sync(0xFFFFFFFFu, incl, 31);
    const double excl = incl - seg;
    const double tt = static_cast<double>(u) * W;
    const unsigned hit = __ballot_sync(0xFFFFFFFFu, incl > tt && seg > 0.0);
    int step = -1;
    double trel = 0.0;
    if (hit) {
      const int first = __ffs(hit) - 1;
      if (lane == first) {
        double acc = excl;
        for (int st = s0; st < s1; ++st) {
          const double x = static_cast<double>(step_tot[st]);
          if (acc + x > tt && x > 0.0) {
            step = st;
            trel = tt - acc;
            break;
          }
          acc += x;
        }
        if (step < 0) {
          step = lastpos;
          trel = INFINITY;
        }
      }
      step = __shfl_sync(0xFFFFFFFFu, step, first);
      trel = __shfl_sync(0xFFFFFFFFu, trel, first);
    } else {
      step = warp_max_i(lastpos);
      trel = INFINITY;
    }
    if (lane == 0) {
      ctl.W = W;
      ctl.step = step;
      ctl.t_rel = trel;
    }
  }
  draw_sync();
  Wout = ctl.W;
  int token = -1;
  margin = 0.f;
  if (w == 0 && ctl.step >= 0) {
    const int st = ctl.step;
    const bool exact = ctl.t_rel != INFINITY;
    const float tr = static_cast<float>(ctl.t_rel);
    const int base = st * kPStep + lane * 8;
    float x[8];
    step_weights<TE>(gp, gq, dp, dq, residual, base, V, x);
    float s = 0.f;
    int lp = -1;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      s += x[e];
      if (x[e] > 0.f) lp = base + e;
    }
    float incl = s;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float y = __shfl_up_sync(0xFFFFFFFFu, incl, off);
      if (lane >= off) incl += y;
    }
    const float excl = incl - s;
    const unsigned hit = exact ? __ballot_sync(0xFFFFFFFFu, incl > tr && s > 0.f) : 0u;
    if (hit) {
      const int first = __ffs(hit) - 1;
      int found = -1;
      float mg = 0.f;
      if (lane == first) {
        float run = excl;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float prev = run;
          run += x[e];
          if (found < 0 && x[e] > 0.f && run > tr) {
            found = base + e;
            mg = fminf(tr - prev, run - tr);
          }
        }
        if (found < 0) found = lp;
      }
      token = __shfl_sync(0xFFFFFFFFu, found, first);
      margin = __shfl_sync(0xFFFFFFFFu, mg, first);
    } else {
      token = warp_max_i(lp);
      margin = 0.f;
    }
    if (lane == 0) ctl.step = token;  // hand the token to the group
  }
  draw_sync();
  token = ctl.step;
  draw_sync();
  return token;
}

// ---------------------------------------------------------------------------
// distributed draws
// ---------------------------------------------------------------------------
//
// A sequence's final draw is split into weight jobs: job k of wj sums the
// draw weights of steps [k wj_steps, (k + 1) wj_steps) (256 entries each) into
// the sequence's step-total array.  Job (s, k) belongs to the draw group of
// CTA (s + 1 + k wj_stride) mod G, so one group's jobs come from sequences
// far apart and the jobs of one draw run side by side in wj groups.  The
// sequence's owner searches once the job count is complete: a double-
// precision prefix over the step totals finds the step, one warp scans it.
// Draws whose single-precision search lands within the refine guard of a
// boundary are queued for the precise redraw: per queued draw, pj jobs of
// double-float step sums and normaliser shares, claimed by groups with no
// other work left; the last job searches in double precision and overwrites
// the token.

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_i32(int *p, int v) {
  asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

constexpr int kSeqWords = sizeof(PassSeq) / 4;
static_assert(kSeqWords <= 32, "a descriptor is published by one warp");
constexpr unsigned long long kTag = 1ull << 32;  // marks a written 64-bit entry

// Publish ctl.ps as sequence s's descriptor: one 32-bit word per tagged
// 64-bit entry, so a reader can tell a complete descriptor without a fence
// (draw group; ctl.ps must be visible to the group).
__device__ __forceinline__ void publish_seq(const Params &P, PassCtl &ctl, int s) {
  const int t = threadIdx.x - kPDrawWarp0 * 32;
  if (t < kSeqWords) {
    const uint32_t v = reinterpret_cast<const uint32_t *>(&ctl.ps)[t];
    P.pseqw[static_cast<long long>(s) * kSeqWords + t] = static_cast<unsigned long long>(v) | kTag;
  }
}

// Copy sequence s's descriptor into shared memory (draw group), reading again
// while any entry is still unset.  Returns false (in every thread) when the
// bounded wait gave up: the scratch then holds no usable descriptor.
__device__ bool load_seq(const Params &P, PassCtl &ctl, int s) {
  const int t = threadIdx.x - kPDrawWarp0 * 32;
  if (t == 0) ctl.redo = 1;
  if (t < 32) {
    const unsigned long long *src = P.pseqw + static_cast<long long>(s) * kSeqWords;
    uint32_t *dst = reinterpret_cast<uint32_t *>(&ctl.ps);
    const long long t0 = pass_ns();
    while (true) {
      bool ok = true;
      if (t < kSeqWords) {
        const unsigned long long v = __ldcg(src + t);
        ok = (v >> 32) != 0ull;
        dst[t] = static_cast<uint32_t>(v);
      }
      if (__all_sync(0xFFFFFFFFu, ok)) break;
      if (pass_ns() - t0 > kPPollLimitNs) {
        if (t == 0) {
          atomicOr(P.err, 1u);
          ctl.redo = 0;
        }
        break;
      }
      __nanosleep(100);
    }
  }
  draw_sync();
  const bool good = ctl.redo != 0;
  draw_sync();
  return good;
}

// Rows of a sequence's draw position j.
template <typename TE>
__device__ __forceinline__ void draw_rows(const Params &P, int s, int j, const TE *&gp,
                                          const TE *&gq) {
  gp = static_cast<const TE *>(
      row_ptr(P.target, static_cast<long long>(s) * (P.gamma + 1) + j, P.ld_t, sizeof(TE)));
  gq = static_cast<const TE *>(row_ptr(
      P.draft, static_cast<long long>(s) * P.gamma + (j < P.gamma ? j : 0), P.ld_d, sizeof(TE)));
}

// Outputs of a finished draw and the unit record the residual output reads.
__device__ void write_final(const Params &P, int s, const PassSeq &ps, int token, double W,
                            int near) {
  const long long obase = static_cast<long long>(s) * (P.gamma + 1);
  const long long unit = obase + ps.j;
  uint32_t flags = ps.flags;
  flags |= *reinterpret_cast<const volatile uint32_t *>(P.err) ? SPEC_FLAG_TIMEOUT : 0u;
  P.out_tokens[obase + ps.j] = token;
  P.out_num[s] = ps.j;
  if (P.out_flags) P.out_flags[s] = flags;
  UnitOut o;
  o.next = -1;
  o.token = token;
  o.flags = flags;
  o.near = near;
  P.outs[unit] = o;
  UnitStats st;
  st.p = ps.dp;
  st.q = ps.dq;
  st.c = ps.residual ? 1.f : 0.f;
  st.total = static_cast<float>(W);
  st.kind = ps.kind;
  st.node = ps.j;
  st.n_res = ps.residual;
  st.pad = 0;
  P.stats[unit] = st;
  P.final_unit[s] = static_cast<int>(unit);
}

// One more sequence is final (single thread; a count only, the outputs are
// read after the kernel).
__device__ __forceinline__ void count_final(const Params &P) {
  asm volatile("red.relaxed.gpu.global.add.u32 [%0], 1;" ::"l"(P.pctr + 2) : "memory");
}

// Decide sequence s: merge its records into the row statistics, run the
// acceptance tests, and publish the draw (or finish the sequence when the
// token needs no draw).
template <typename TE>
__device__ void decide(const Params &P, PassCtl &ctl, int seq) {
  const int t = threadIdx.x - kPDrawWarp0 * 32, lane = t & 31, w = t >> 5;
  const int gamma = P.gamma, rps = 2 * gamma + 1, V = P.V;
  const float Tp = __ldg(P.Tp + seq), Tq = __ldg(P.Tq + seq);
  const bool p_arg = row_is_arg(Tp), q_arg = row_is_arg(Tq);
  const bool tp_bad = !(Tp >= 0.f) || Tp == INFINITY, tq_bad = !(Tq >= 0.f) || Tq == INFINITY;
  const float kp = p_arg ? 0.f : kLog2e / Tp, kq = q_arg ? 0.f : kLog2e / Tq;
  // 1. row statistics (the progress count can run ahead of the records:
  // merge again while any still reads zero)
  {
    const long long t0 = pass_ns();
    // the draft tokens, loaded beside the records
    const int xtok = t < gamma ? __ldg(P.tokens + static_cast<long long>(seq) * gamma + t) : 0;
    while (true) {
      if (merge_rows(P, ctl, seq, p_arg, q_arg, kp, kq)) {
        if (t < gamma) ctl.tokx[t] = xtok;
        break;
      }
      if (pass_ns() - t0 > kPPollLimitNs) {
        if (t == 0) atomicOr(P.err, 1u);
        break;
      }
      __nanosleep(200);
    }
  }
  if (t < rps) {  // one thread per row
    const int r = t;
    const bool draft = r > gamma;
    const bool arg = draft ? q_arg : p_arg;
    const bool tbad = draft ? tq_bad : tp_bad;
    const PassRow pr = ctl.row[r];
    RowDesc d;
    d.thr = -INFINITY;
    d.flags = 0u;
    d.m = 0.f;
    d.k = d.nmk = d.invS = 0.f;
    d.a = 0;
    if (arg) {
      d.onehot = 1;
      d.a = pr.a;
      if (tbad || pr.bad) d.flags = SPEC_FLAG_NONFINITE;
    } else if (pr.bad) {
      d.onehot = 1;  // the finite argmax is filled in below
      d.flags = SPEC_FLAG_NONFINITE;
    } else {
      const float kk = draft ? kq : kp;
      d.onehot = 0;
      d.k = kk;
      d.m = pr.m;
      d.nmk = -pr.m * kk;
      d.invS = 1.f / pr.S;
    }
    ctl.desc[r] = d;
  }
  draw_sync();
  for (int r = 0; r < rps; ++r) {  // rows whose sampling statistics were not finite (rare)
    const bool draft = r > gamma;
    if ((draft ? q_arg : p_arg) || !ctl.row[r].bad) continue;
    const long long row = draft ? static_cast<long long>(seq) * gamma + (r - gamma - 1)
                                : static_cast<long long>(seq) * (gamma + 1) + r;
    const TE *g = static_cast<const TE *>(
        row_ptr(draft ? P.draft : P.target, row, draft ? P.ld_d : P.ld_t, sizeof(TE)));
    const int a = finite_argmax_row<TE>(g, V, ctl);
    if (t == 0) ctl.desc[r].a = a;
  }
  draw_sync();
  // 2. acceptance tests, one lane per draft position
  if (w == 0) {
    int i = lane;
    uint32_t f = 0u;
    bool reject = true;
    if (i < gamma) {
      const RowDesc dp = ctl.desc[i];
      const RowDesc dq = ctl.desc[gamma + 1 + i];
      const int x = ctl.tokx[i];
      f = dp.flags;
      const bool valid = x >= 0 && x < V;
      if (!valid) f |= SPEC_FLAG_BAD_TOKEN;
      if (dp.onehot) {
        reject = !(valid && x == dp.a);
      } else {
        f |= dq.flags;
        if (valid) {
          const TE *gp = static_cast<const TE *>(
              row_ptr(P.target, static_cast<long long>(seq) * (gamma + 1) + i, P.ld_t,
                      sizeof(TE)));
          const TE *gq = static_cast<const TE *>(
              row_ptr(P.draft, static_cast<long long>(seq) * gamma + i, P.ld_d, sizeof(TE)));
          const float px = pprob(dp, dp.onehot ? 0.f : to_f32(gp[x]), x);
          const float qx = pprob(dq, dq.onehot ? 0.f : to_f32(gq[x]), x);
          if (!(qx > 0.f)) {
            f |= SPEC_FLAG_ZERO_Q;
          } else {
            const float uu = unit_uniform(P, seq, i, 0);
            reject = !(uu < fminf(1.f, px / qx));
          }
        }
      }
      ctl.pos_flags[i] = static_cast<int>(f);
    }
    const unsigned rej = __ballot_sync(0xFFFFFFFFu, reject && i < gamma);
    const int j = rej ? __ffs(rej) - 1 : gamma;
    // the draw uniform at every position, computed beside the tests
    const float ud = i <= gamma ? unit_uniform(P, seq, i, 1) : 0.f;
    const float u_draw = __shfl_sync(0xFFFFFFFFu, ud, j);
    uint32_t fo = (i < j) ? f : 0u;
    fo = warp_or(fo);
    if (lane == 0) {
      if (j < gamma) fo |= static_cast<uint32_t>(ctl.pos_flags[j]);
      else fo |= ctl.desc[gamma].flags;
      ctl.j = j;
      ctl.flags = fo;
      ctl.u_draw = u_draw;
    }
  }
  draw_sync();
  const int j = ctl.j;
  const long long obase = static_cast<long long>(seq) * (gamma + 1);
  for (int i = t; i <= gamma; i += kPDrawThreads) {
    if (i < j) P.out_tokens[obase + i] = __ldg(P.tokens + static_cast<long long>(seq) * gamma + i);
    else if (i > j) P.out_tokens[obase + i] = -1;
  }
  // 3. the draw at j
  if (t == 0) {
    PassSeq ps;
    ps.dp = ctl.desc[j];
    ps.residual = j < gamma ? 1 : 0;
    if (ps.residual) {
      ps.dq = ctl.desc[gamma + 1 + j];
    } else {
      ps.dq = ps.dp;
      ps.dq.onehot = 1;
      ps.dq.a = 0;
    }
    ps.j = j;
    ps.flags = ctl.flags;
    ps.W = 0.f;
    ps.u = 0.f;
    if (ps.dp.onehot) {
      ps.kind = j < gamma ? 1 : 0;
      ps.residual = 0;
      ps.draw = 0;
      write_final(P, seq, ps, ps.dp.a, 0.0, 0);
      count_final(P);
    } else {
      ps.kind = j < gamma ? 2 : 0;
      ps.u = ctl.u_draw;
      ps.draw = 1;
    }
    ctl.ps = ps;
  }
  draw_sync();
  publish_seq(P, ctl, seq);  // the weight jobs read it (and skip when no draw)
  if (t == 0) {
    ctl.ps_own = ctl.ps;
    ctl.next_srch = ctl.ps.draw ? seq : -1;
  }
  draw_sync();
}

// Single-precision inverse-CDF search over sequence s's published step
// totals, then the scan of the owning step (draw group; ctl.ps holds the
// descriptor).  Finishes the sequence or queues it for the precise redraw.
template <typename TE>
__device__ void fsearch(const Params &P, PassCtl &ctl, float *step_tot, int s) {
  const int t = threadIdx.x - kPDrawWarp0 * 32, lane = t & 31, w = t >> 5;
  const int nsteps = P.steps, V = P.V;
  const unsigned long long *fst = P.fstep + static_cast<long long>(s) * nsteps;
  PassSeq ps = ctl.ps_own;
  const TE *gp, *gq;
  draw_rows<TE>(P, s, ps.j, gp, gq);
  if (w == 0) {
    const int per = (nsteps + 31) / 32;
    const int s0 = min(nsteps, lane * per), s1 = min(nsteps, s0 + per);
    double seg = 0.0;
    int lastpos = -1;
    const long long t0 = pass_ns();
    while (true) {  // read again while a job's totals are not all visible
      bool miss = false;
      seg = 0.0;
      lastpos = -1;
      for (int b0 = s0; b0 < s1; b0 += 16) {  // sixteen loads in flight
        unsigned long long x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = b0 + i < s1 ? __ldcg(fst + b0 + i) : kTag;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          miss |= (x[i] >> 32) == 0ull;
          const float v = __uint_as_float(static_cast<uint32_t>(x[i]));
          seg += static_cast<double>(v);
          if (v > 0.f) lastpos = b0 + i;
        }
      }
      if (!__any_sync(0xFFFFFFFFu, miss)) break;
      if (pass_ns() - t0 > kPPollLimitNs) {
        if (lane == 0) atomicOr(P.err, 1u);
        break;
      }
      __nanosleep(100);
    }
    double incl = seg;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const double y = __shfl_up_sync(0xFFFFFFFFu, incl, off);
      if (lane >= off) incl += y;
    }
    const double W = __shfl_sync(0xFFFFFFFFu, incl, 31);
    const double tt = static_cast<double>(ps.u) * W;
    const unsigned hit = __ballot_sync(0xFFFFFFFFu, incl > tt && seg > 0.0);
    int step = -1;
    double trel = 0.0;
    if (hit) {
      const int first = __ffs(hit) - 1;
      if (lane == first) {
        double acc = incl - seg;
        for (int b0 = s0; b0 < s1 && step < 0; b0 += 16) {
          float xs[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            xs[i] = b0 + i < s1 ? __uint_as_float(static_cast<uint32_t>(__ldcg(fst + b0 + i))) : 0.f;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const double x = static_cast<double>(xs[i]);
            if (step < 0 && b0 + i < s1) {
              if (acc + x > tt && x > 0.0) {
                step = b0 + i;
                trel = tt - acc;
              }
              acc += x;
            }
          }
        }
        if (step < 0) {
          step = lastpos;
          trel = INFINITY;
        }
      }
      step = __shfl_sync(0xFFFFFFFFu, step, first);
      trel = __shfl_sync(0xFFFFFFFFu, trel, first);
    } else {
      step = warp_max_i(lastpos);
      trel = INFINITY;
    }
    int token = -1;
    float margin = 0.f;
    if (step >= 0) {
      const bool exact = trel != INFINITY;
      const float tr = static_cast<float>(trel);
      const int base = step * kPStep + lane * 8;
      float x[8];
      step_weights<TE>(gp, gq, ps.dp, ps.dq, ps.residual, base, V, x);
      float sm = 0.f;
      int lp = -1;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        sm += x[e];
        if (x[e] > 0.f) lp = base + e;
      }
      float fin = sm;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xFFFFFFFFu, fin, off);
        if (lane >= off) fin += y;
      }
      const float excl = fin - sm;
      const unsigned h2 = exact ? __ballot_sync(0xFFFFFFFFu, fin > tr && sm > 0.f) : 0u;
      if (h2) {
        const int first = __ffs(h2) - 1;
        int found = -1;
        float mg = 0.f;
        if (lane == first) {
          float run = excl;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float prev = run;
            run += x[e];
            if (found < 0 && x[e] > 0.f && run > tr) {
              found = base + e;
              mg = fminf(tr - prev, run - tr);
            }
          }
          if (found < 0) found = lp;
        }
        token = __shfl_sync(0xFFFFFFFFu, found, first);
        margin = __shfl_sync(0xFFFFFFFFu, mg, first);
      } else {
        token = warp_max_i(lp);
        margin = 0.f;
      }
    }
    if (lane == 0) {
      ctl.W = W;
      ctl.step = token;
      ctl.red_v[0] = margin;
    }
  }
  draw_sync();
  int token = ctl.step;
  double W = ctl.W;
  float margin = ctl.red_v[0];
  draw_sync();
  if (ps.residual && !(W > 0.0)) {
    // degenerate residual: draw from p itself (this group alone)
    ps.flags |= SPEC_FLAG_DEGENERATE_RESIDUAL;
    ps.residual = 0;
    ps.dq = ps.dp;
    ps.dq.onehot = 1;
    ps.dq.a = 0;
    token = pass_draw<TE>(P, ctl, step_tot, gp, gq, ps.dp, ps.dq, 0, ps.u, margin, W);
  }
  // redraw precisely when the draw came within 1e-6 of the draw mass of a
  // boundary (the single-precision boundary error measured on 128K-entry rows
  // stays below 3e-7 of it)
  const int near = margin < 1e-6f * static_cast<float>(W) ? 1 : 0;
  if (t == 0) {
    ps.W = static_cast<float>(W);
    write_final(P, s, ps, token, W, near);
    if (!near) count_final(P);
    ctl.ps = ps;
    ctl.redo = near;
  }
  draw_sync();
  if (ctl.redo) {
    // the precise redraw reads the final descriptor (a rare path: fenced)
    publish_seq(P, ctl, s);
    draw_sync();
    if (t == 0) {
      __threadfence();
      const uint32_t i = atomicAdd(P.pctr, 1u);
      st_release_i32(P.near_list + i, s + 1);
    }
    draw_sync();
  }
}

// Weight job (s, k): step totals of steps [k kf_steps, (k + 1) kf_steps).
template <typename TE>
__device__ void fjob(const Params &P, PassCtl &ctl, float *step_tot, int s, int k) {
  const int t = threadIdx.x - kPDrawWarp0 * 32, lane = t & 31, w = t >> 5;
  const PassSeq &ps = ctl.ps;  // read by the scheduler
  const TE *gp, *gq;
  draw_rows<TE>(P, s, ps.j, gp, gq);
  const RowDesc dp = ps.dp, dq = ps.dq;
  const int residual = ps.residual;
  const int V = P.V;
  const int b0 = k * P.wj_steps, b1 = min(P.steps, b0 + P.wj_steps);
  unsigned long long *fst = P.fstep + static_cast<long long>(s) * P.steps;
  // full steps four per warp at a time, their loads issued before any is used
  constexpr int kU = 4;
  const int nfull = min(b1, V / kPStep);
  int st0 = b0 + w;
  for (; st0 + (kU - 1) * kPDrawWarps < nfull; st0 += kPDrawWarps * kU) {
    Raw8<TE> rp[kU], rq[kU];
#pragma unroll
    for (int q = 0; q < kU; ++q) {
      const int base = (st0 + q * kPDrawWarps) * kPStep + lane * 8;
      rp[q].load(gp + base);
      if (residual) rq[q].load(gq + base);
    }
#pragma unroll
    for (int q = 0; q < kU; ++q) {
      const int base = (st0 + q * kPDrawWarps) * kPStep + lane * 8;
      float zp[8], zq[8], x[8];
      rp[q].get(zp);
      rq[q].get(zq);
      weights8(dp, dq, residual, base, zp, zq, x);
      float sm = ((x[0] + x[1]) + (x[2] + x[3])) + ((x[4] + x[5]) + (x[6] + x[7]));
      sm = warp_sum(sm);
      if (lane == 0) fst[st0 + q * kPDrawWarps] = static_cast<unsigned long long>(__float_as_uint(sm)) | kTag;
    }
  }
  for (int st = st0; st < b1; st += kPDrawWarps) {
    float x[8];
    step_weights<TE>(gp, gq, dp, dq, residual, st * kPStep + lane * 8, V, x);
    float sm = ((x[0] + x[1]) + (x[2] + x[3])) + ((x[4] + x[5]) + (x[6] + x[7]));
    sm = warp_sum(sm);
    if (lane == 0) fst[st] = static_cast<unsigned long long>(__float_as_uint(sm)) | kTag;
  }
  draw_sync();
  // count the job (relaxed): the sequence's owner searches once the count is
  // complete, reading the totals again until every job's entries are visible
  if (t == 0) asm volatile("red.relaxed.gpu.global.add.u32 [%0], 1;" ::"l"(P.sctr + 4ll * s + 1)
                           : "memory");
}

// Double-float weights of the 8 entries from `base` (precise redraw).
template <typename TE>
__device__ __forceinline__ void pweights8(const TE *gp, const TE *gq, const HpRow &rp,
                                          const HpRow &rq, int residual, Df rho, int base, int V,
                                          bool vec, const PassCtl &ctl, Df w[8]) {
  float zp[8], zq[8];
  hp_load8<TE>(gp, base, V, vec, zp);
  if (residual) hp_load8<TE>(gq, base, V, vec, zq);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const Df ep = hp_exp(rp, zp[e], ctl.tab_hi, ctl.tab_lo);
    if (!residual || ep.hi == 0.f) {
      w[e] = ep;
      continue;
    }
    const Df eq = hp_exp(rq, zq[e], ctl.tab_hi, ctl.tab_lo);
    const Df d = df_sub(ep, df_mul(rho, eq));
    w[e] = d.hi > 0.f ? d : Df{0.f, 0.f};
  }
}

// Sum over the pj normaliser shares of sequence s (the same bits in every
// lane and every group: lane-strided sums, a butterfly, lane 0's value).
__device__ __forceinline__ double pshare_sum(const Params &P, int s, int which) {
  const int lane = threadIdx.x & 31;
  const double *x = P.ppart + static_cast<long long>(s) * P.pj * 2 + which;
  double v = 0.0;
  for (int k = lane; k < P.pj; k += 32) v += __ldcg(x + 2 * k);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
  return __shfl_sync(0xFFFFFFFFu, v, 0);
}

// Double-precision search of a precise redraw (the group that completed the
// draw's jobs).  The step totals are A - rho B with rho = S_p / S_q from the
// normaliser shares (A alone for a draw from p); steps a job marked
// uncertain are first recomputed entry by entry.  One warp then finds the
// step by a prefix over its lanes' runs of steps and scans it with double-
// float weights; the token is overwritten.
template <typename TE>
__device__ void psearch(const Params &P, PassCtl &ctl, int s, const TE *gp, const TE *gq,
                        const HpRow &rp, const HpRow &rq, bool vec) {
  const int t = threadIdx.x - kPDrawWarp0 * 32, lane = t & 31, w = t >> 5;
  const PassSeq &ps = ctl.ps;
  const int nsteps = P.steps;
  double *pa = P.pstep + static_cast<long long>(s) * 2 * nsteps;
  double *pb = pa + nsteps;
  double rhod = 0.0;
  Df rho{0.f, 0.f};
  if (ps.residual) {
    const double Sp = pshare_sum(P, s, 0), Sq = pshare_sum(P, s, 1);
    rhod = Sp / Sq;
    rho = df_from_double(rhod);
  }
  if (t == 0) ctl.redo = static_cast<int>(__ldcg(P.sctr + 4ll * s + 3));
  draw_sync();
  if (ctl.redo) {
    // uncertain steps: their exact totals, one warp per step
    for (int base = w * 32; base < nsteps; base += kPDrawWarps * 32) {
      const int st = base + lane;
      unsigned todo = __ballot_sync(0xFFFFFFFFu, st < nsteps && __ldcg(pb + st) < 0.0);
      while (todo) {
        const int x = base + __ffs(todo) - 1;
        todo &= todo - 1;
        Df wd[8];
        pweights8<TE>(gp, gq, rp, rq, ps.residual, rho, x * kPStep + lane * 8, P.V, vec, ctl, wd);
        Df acc{0.f, 0.f};
#pragma unroll
        for (int e = 0; e < 8; ++e) acc = df_add(acc, wd[e]);
        double v = df_to_double(acc);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
        if (lane == 0) {
          pa[x] = v;
          pb[x] = 0.0;
        }
      }
    }
    __threadfence_block();
    draw_sync();
  }
  if (w == 0) {
    const int per = (nsteps + 31) / 32;
    const int s0 = min(nsteps, lane * per), s1 = min(nsteps, s0 + per);
    double seg = 0.0;
    int lastpos = -1;
    for (int b0 = s0; b0 < s1; b0 += 8) {  // eight pairs of loads in flight
      double xa[8], xb[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        xa[i] = b0 + i < s1 ? __ldcg(pa + b0 + i) : 0.0;
        xb[i] = b0 + i < s1 ? __ldcg(pb + b0 + i) : 0.0;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const double x = xa[i] - rhod * xb[i];
        seg += x;
        if (x > 0.0) lastpos = b0 + i;
      }
    }
    double incl = seg;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const double y = __shfl_up_sync(0xFFFFFFFFu, incl, off);
      if (lane >= off) incl += y;
    }
    const double Z = __shfl_sync(0xFFFFFFFFu, incl, 31);
    const double tt = static_cast<double>(ps.u) * Z;
    const unsigned hit = __ballot_sync(0xFFFFFFFFu, incl > tt && seg > 0.0);
    int step = -1;
    double trel = 0.0;
    if (hit) {
      const int first = __ffs(hit) - 1;
      if (lane == first) {
        double acc = incl - seg;
        for (int b0 = s0; b0 < s1 && step < 0; b0 += 8) {
          double xs[8];
#pragma unroll
          for (int i = 0; i < 8; ++i)
            xs[i] = b0 + i < s1 ? __ldcg(pa + b0 + i) - rhod * __ldcg(pb + b0 + i) : 0.0;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (step < 0 && b0 + i < s1) {
              if (acc + xs[i] > tt && xs[i] > 0.0) {
                step = b0 + i;
                trel = tt - acc;
              }
              acc += xs[i];
            }
          }
        }
        if (step < 0) {
          step = lastpos;
          trel = INFINITY;
        }
      }
      step = __shfl_sync(0xFFFFFFFFu, step, first);
      trel = __shfl_sync(0xFFFFFFFFu, trel, first);
    } else {
      step = warp_max_i(lastpos);
      trel = INFINITY;
    }
    int token = -1;
    if (step >= 0) {
      const int base = step * kPStep + lane * 8;
      Df wd[8];
      pweights8<TE>(gp, gq, rp, rq, ps.residual, rho, base, P.V, vec, ctl, wd);
      double x[8];
      double sm = 0.0;
      int lp = -1;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        x[e] = df_to_double(wd[e]);
        sm += x[e];
        if (x[e] > 0.0) lp = base + e;
      }
      double fin = sm;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const double y = __shfl_up_sync(0xFFFFFFFFu, fin, off);
        if (lane >= off) fin += y;
      }
      const unsigned h2 =
          trel != INFINITY ? __ballot_sync(0xFFFFFFFFu, fin > trel && sm > 0.0) : 0u;
      if (h2) {
        const int first = __ffs(h2) - 1;
        int found = -1;
        if (lane == first) {
          double run = fin - sm;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            run += x[e];
            if (found < 0 && x[e] > 0.0 && run > trel) found = base + e;
          }
          if (found < 0) found = lp;
        }
        token = __shfl_sync(0xFFFFFFFFu, found, first);
      } else {
        token = warp_max_i(lp);
      }
    }
    if (lane == 0) {
      if (token >= 0) {
        const long long obase = static_cast<long long>(s) * (P.gamma + 1);
        P.out_tokens[obase + ps.j] = token;
        P.outs[obase + ps.j].token = token;
      }
      count_final(P);
    }
  }
  draw_sync();
}

// Precise job v: redraw item v / pj, slice v % pj of its steps.  For each
// 256-entry step of the slice it stores the double-float sums A of e_p and B
// of e_q over the entries whose weight e_p - rho e_q is certainly positive,
// classified with the single-precision rho of the row statistics (within
// 1e-6 of the exact one; an entry is certain when |e_p - rho e_q| > 1e-5 e_p),
// or B = -1 when an entry of the step is uncertain; and the slice's shares of
// S_p and S_q.  A draw from p stores A = the sum of e_p, B = 0.  The job that
// completes the item's count searches.
template <typename TE>
__device__ void pjob(const Params &P, PassCtl &ctl, int v) {
  const int t = threadIdx.x - kPDrawWarp0 * 32, lane = t & 31, w = t >> 5;
  const int kp = P.pj;
  const int item = v / kp, k = v - item * kp;
  if (t == 0) {
    const long long t0 = pass_ns();
    int sv1;
    while ((sv1 = *reinterpret_cast<const volatile int *>(P.near_list + item)) == 0) {
      if (pass_ns() - t0 > kPPollLimitNs) {
        atomicOr(P.err, 1u);
        break;
      }
      __nanosleep(100);
    }
    __threadfence();
    ctl.job_s = sv1 - 1;
  }
  draw_sync();
  const int s = ctl.job_s;
  if (s < 0 || s >= P.nseq || !load_seq(P, ctl, s)) return;
  const PassSeq &ps = ctl.ps;
  if (ps.j < 0 || ps.j > P.gamma) return;  // not a drawn position: never use it as a row
  const TE *gp, *gq;
  draw_rows<TE>(P, s, ps.j, gp, gq);
  const bool vec = ((reinterpret_cast<uintptr_t>(gp) | reinterpret_cast<uintptr_t>(gq)) & 15u) == 0;
  const HpRow rp = hp_row(ps.dp, __ldg(P.Tp + s));
  const HpRow rq = ps.residual ? hp_row(ps.dq, __ldg(P.Tq + s)) : rp;
  const int residual = ps.residual;
  const float rho_a = residual ? ps.dq.invS / ps.dp.invS : 0.f;  // S_p / S_q, single precision
  const int V = P.V;
  const int b0 = k * P.pj_steps, b1 = min(P.steps, b0 + P.pj_steps);
  double *pa = P.pstep + static_cast<long long>(s) * 2 * P.steps;
  double *pb = pa + P.steps;
  uint32_t *cnt = P.sctr + 4ll * s;
  double sp_tot = 0.0, sq_tot = 0.0;
  bool unc_any = false;
  for (int st = b0 + w; st < b1; st += kPDrawWarps) {
    const int base = st * kPStep + lane * 8;
    float zp[8], zq[8];
    hp_load8<TE>(gp, base, V, vec, zp);
    if (residual) hp_load8<TE>(gq, base, V, vec, zq);
    Df sp{0.f, 0.f}, sq{0.f, 0.f}, a{0.f, 0.f}, b{0.f, 0.f};
    bool unc = false;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const Df ep = hp_exp(rp, zp[e], ctl.tab_hi, ctl.tab_lo);
      sp = df_add(sp, ep);
      if (!residual) continue;
      const Df eq = hp_exp(rq, zq[e], ctl.tab_hi, ctl.tab_lo);
      sq = df_add(sq, eq);
      if (ep.hi > 0.f) {
        const float d = fmaf(-rho_a, eq.hi, ep.hi);
        if (d > 1e-5f * ep.hi) {
          a = df_add(a, ep);
          b = df_add(b, eq);
        } else if (d >= -1e-5f * ep.hi) {
          unc = true;
        }
      }
    }
    double A = residual ? df_to_double(a) : df_to_double(sp);
    double Bq = df_to_double(b);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      A += __shfl_xor_sync(0xFFFFFFFFu, A, off);
      Bq += __shfl_xor_sync(0xFFFFFFFFu, Bq, off);
    }
    unc = __any_sync(0xFFFFFFFFu, unc);
    if (lane == 0) {
      pa[st] = A;
      pb[st] = unc ? -1.0 : Bq;
    }
    unc_any |= unc;
    sp_tot += df_to_double(sp);
    sq_tot += df_to_double(sq);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    sp_tot += __shfl_xor_sync(0xFFFFFFFFu, sp_tot, off);
    sq_tot += __shfl_xor_sync(0xFFFFFFFFu, sq_tot, off);
  }
  if (lane == 0) {
    ctl.pred[0][w] = sp_tot;
    ctl.pred[1][w] = sq_tot;
    ctl.red_i[w] = unc_any ? 1 : 0;
  }
  draw_sync();
  if (t == 0) {
    double A = 0.0, B = 0.0;
    int u = 0;
    for (int x = 0; x < kPDrawWarps; ++x) {
      A += ctl.pred[0][x];
      B += ctl.pred[1][x];
      u |= ctl.red_i[x];
    }
    double *dst = P.ppart + (static_cast<long long>(s) * kp + k) * 2;
    dst[0] = A;
    dst[1] = B;
    if (u) atomicAdd(cnt + 3, 1u);
    __threadfence();
    const uint32_t old = atomicAdd(cnt + 2, 1u);
    ctl.redo = old + 1 == static_cast<uint32_t>(kp) ? 1 : 0;
    if (ctl.redo) __threadfence();
  }
  draw_sync();
  if (ctl.redo) psearch<TE>(P, ctl, s, gp, gq, rp, rq, vec);
}

// Weight jobs of group g: job (s, k) belongs to group (s + 1 + k stride) mod G,
// so the group's jobs are the sequences s = (g - 1 - k stride) mod G + m G.
// The wj residues are sorted once (ctl.fj_s / fj_k, warp 0); the m-th pass
// over them gives the jobs in sequence order.
__device__ void init_fjobs(const Params &P, PassCtl &ctl, int g, int G) {
  const int lane = threadIdx.x & 31;
  int r = INT_MAX, k = lane;
  if (lane < P.wj) {
    r = (g - 1 - lane * P.wj_stride) % G;
    if (r < 0) r += G;
  }
  // rank of each residue among the lanes (residues are distinct)
  int rank = 0;
  for (int x = 0; x < 32; ++x) {
    const int rx = __shfl_sync(0xFFFFFFFFu, r, x);
    rank += rx < r ? 1 : 0;
  }
  if (lane < P.wj) {
    ctl.fj_s[rank] = r;
    ctl.fj_k[rank] = k;
  }
  if (lane == 0) {
    ctl.fj_i = 0;
    ctl.fj_m = 0;
  }
  __syncwarp();
}

// Advance to the group's next weight job (thread 0): ctl.next_f / next_k, or
// next_f = nseq when none is left.
__device__ void advance_fjob(const Params &P, PassCtl &ctl, int G) {
  int i = ctl.fj_i, m = ctl.fj_m;
  while (true) {
    if (i >= P.wj) {
      i = 0;
      ++m;
    }
    const long long s = ctl.fj_s[i] + static_cast<long long>(m) * G;
    if (s >= P.nseq && i == 0) {  // residues are sorted: this pass and later are empty
      ctl.next_f = P.nseq;
      break;
    }
    if (s < P.nseq) {
      ctl.next_f = static_cast<int>(s);
      ctl.next_k = ctl.fj_k[i];
      ++i;
      break;
    }
    i = P.wj;  // the rest of this pass is past the batch
  }
  ctl.fj_i = i;
  ctl.fj_m = m;
}

// Timed-out sequence: no tokens, SPEC_FLAG_TIMEOUT (single thread).
__device__ void write_timeout(const Params &P, int seq) {
  P.out_num[seq] = 0;
  if (P.out_flags) P.out_flags[seq] = SPEC_FLAG_TIMEOUT;
  P.final_unit[seq] = -1;
  for (int i = 0; i <= P.gamma; ++i) P.out_tokens[static_cast<long long>(seq) * (P.gamma + 1) + i] = -1;
}

enum { kActIdle = 0, kActDecide = 1, kActWeights = 2, kActPrecise = 3, kActExit = 4, kActSearch = 5 };

// The draw group's scheduler: decide owned sequences as their chunks complete,
// run weight jobs as their descriptors appear, and otherwise take precise
// jobs; leave when every sequence of the batch is final.
template <typename TE>
__device__ void draw_loop(const Params &P, PassCtl &ctl, float *step_tot, const Exp2Table &tab) {
  const int t = threadIdx.x - kPDrawWarp0 * 32;
  const int G = gridDim.x, g = blockIdx.x;
  const uint32_t need = static_cast<uint32_t>((2 * P.gamma + 1) * P.cpr);
  if (t < 32) init_fjobs(P, ctl, g, G);
  if (t == 0) {
    ctl.next_dec = g;
    ctl.next_srch = -1;
    ctl.held_v = -1;
    advance_fjob(P, ctl, G);
    ctl.idle_t0 = pass_ns();
  }
  for (int i = t; i < 64; i += kPDrawThreads) {
    ctl.tab_hi[i] = tab.hi[i];
    ctl.tab_lo[i] = tab.lo[i];
  }
  draw_sync();
  unsigned sleep_ns = 64;
  while (true) {
    if (t < 32) {
      // one round trip: the next weight job's descriptor (tagged words), the
      // progress count of the next owned sequence, the precise-job counters
      const int lane = t;
      const int nd = ctl.next_dec, nf = ctl.next_f;
      unsigned long long dw = kTag;
      uint32_t c = 0u;
      if (lane < kSeqWords && nf < P.nseq) dw = __ldcg(P.pseqw + static_cast<long long>(nf) * kSeqWords + lane);
      if (lane == 31 && nd < P.nseq) c = ld_volatile_pass(P.seq_cnt + nd);
      if (lane == 30) c = ld_volatile_pass(P.pctr);
      if (lane == 29) c = ld_volatile_pass(P.pctr + 1);
      if (lane == 28) c = ld_volatile_pass(P.pctr + 2);
      if (lane == 27 && ctl.next_srch >= 0) c = ld_volatile_pass(P.sctr + 4ll * ctl.next_srch + 1);
      const bool desc_ok = __all_sync(0xFFFFFFFFu, (dw >> 32) != 0ull) && nf < P.nseq;
      const uint32_t cnt = __shfl_sync(0xFFFFFFFFu, c, 31);
      const uint32_t nq = __shfl_sync(0xFFFFFFFFu, c, 30);
      const uint32_t claimed = __shfl_sync(0xFFFFFFFFu, c, 29);
      const uint32_t nfinal = __shfl_sync(0xFFFFFFFFu, c, 28);
      const uint32_t jobs_done = __shfl_sync(0xFFFFFFFFu, c, 27);
      const int ns = ctl.next_srch;
      int act = kActIdle;
      if (ns >= 0 && jobs_done >= static_cast<uint32_t>(P.wj)) {
        act = kActSearch;
      } else if (ns < 0 && nd < P.nseq && cnt >= need) {
        act = kActDecide;
      } else if (desc_ok) {
        act = kActWeights;
        if (lane < kSeqWords) reinterpret_cast<uint32_t *>(&ctl.ps)[lane] = static_cast<uint32_t>(dw);
      } else if (lane == 0) {
        // precise jobs once this group's own decides and weight jobs are done:
        // claim a job id (fetch-and-add), run it once its redraw is queued
        const bool free = ns < 0 && nd >= P.nseq && nf >= P.nseq;
        const uint32_t per_item = static_cast<uint32_t>(P.pj);
        if (free && ctl.held_v < 0 && claimed < nq * per_item)
          ctl.held_v = static_cast<int>(atomicAdd(P.pctr + 1, 1u));
        if (free && ctl.held_v >= 0 && static_cast<uint32_t>(ctl.held_v) < nq * per_item) {
          act = kActPrecise;
          ctl.job_v = ctl.held_v;
          ctl.held_v = -1;
        } else if (free && nfinal >= static_cast<uint32_t>(P.nseq)) {
          act = kActExit;  // every sequence is final: a held id has no job
        } else if (pass_ns() - ctl.idle_t0 > kPPollLimitNs) {
          // nothing moved for too long: give up, marking what this group owns
          atomicOr(P.err, 1u);
          for (int x = nd; x < P.nseq; x += G) write_timeout(P, x);
          act = kActExit;
        }
      }
      if (lane == 0) {
        if (act != kActIdle) ctl.idle_t0 = pass_ns();
        ctl.act = act;
      }
    }
    draw_sync();
    const int act = ctl.act;
    if (act == kActExit) break;
    if (act == kActIdle) {
      if (t == 0) __nanosleep(sleep_ns);
      sleep_ns = min(sleep_ns * 2u, 512u);
      continue;
    }
    sleep_ns = 64;
    if (act == kActSearch) {
      const int s = ctl.next_srch;
      draw_sync();
      fsearch<TE>(P, ctl, step_tot, s);
      if (t == 0) ctl.next_srch = -1;
    } else if (act == kActDecide) {
      const int s = ctl.next_dec;
      draw_sync();
      decide<TE>(P, ctl, s);
      if (t == 0) ctl.next_dec = s + G;
    } else if (act == kActWeights) {
      const int s = ctl.next_f, k = ctl.next_k;
      draw_sync();
      if (ctl.ps.draw) fjob<TE>(P, ctl, step_tot, s, k);
      if (t == 0) advance_fjob(P, ctl, G);
    } else {
      const int v = ctl.job_v;
      draw_sync();
      pjob<TE>(P, ctl, v);
    }
    draw_sync();
  }
}

template <typename TE>
__global__ void __launch_bounds__(kPThreads, 2) pass_kernel(const Params P, const Exp2Table tab) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  PassCtl &ctl = *reinterpret_cast<PassCtl *>(smem_raw);
  unsigned char *ring = smem_raw + P.data_off;
  float *step_tot = reinterpret_cast<float *>(ring + static_cast<size_t>(P.ring) * P.slot_bytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long total =
      static_cast<long long>(P.nseq) * (2 * P.gamma + 1) * static_cast<long long>(P.cpr);
  if (threadIdx.x == 0) {
    for (int s = 0; s < P.ring; ++s) {
      mbar_init(&ctl.full[s], 1);
      mbar_init(&ctl.empty[s], kPConsumerWarps);
      ctl.slot_done[s] = 0;
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();
  if (warp < kPConsumerWarps) {
    consumer_loop<TE>(P, ctl, ring, total);
  } else if (warp == kPProducerWarp) {
    if (lane == 0) producer_loop<TE>(P, ctl, ring, total);
  } else {
    draw_loop<TE>(P, ctl, step_tot, tab);
  }
}

// Job split of the draws for a grid of G CTAs: about 32 weight jobs and 32
// precise jobs per draw, whole 256-entry steps each, at most G weight jobs.
void set_job_split(Params &P, int G) {
  const int steps = P.steps;
  int kf = steps < kPWeightJobs ? steps : kPWeightJobs;
  if (kf > G) kf = G;
  P.wj_steps = (steps + kf - 1) / kf;
  P.wj = (steps + P.wj_steps - 1) / P.wj_steps;
  P.wj_stride = G / P.wj;
  const int kp = steps < kPPreciseJobs ? steps : kPPreciseJobs;
  P.pj_steps = (steps + kp - 1) / kp;
  P.pj = (steps + P.pj_steps - 1) / P.pj_steps;
}

template <typename TE>
cudaError_t launch_pass_t(Params P, const Exp2Table &tab, size_t smem, cudaStream_t stream) {
  // occupancy of the last (device, shared memory) pair, shared by every host
  // thread that launches this instantiation: read and written under the lock
  static std::mutex mu;
  static int cached_dev = -1, cached_smem = -1, cached_blocks = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::unique_lock<std::mutex> lock(mu);
  if (dev != cached_dev || static_cast<int>(smem) != cached_smem) {
    e = cudaFuncSetAttribute(pass_kernel<TE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    int per_sm = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, pass_kernel<TE>, kPThreads, smem);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    cached_blocks = per_sm * sms;
    cached_dev = dev;
    cached_smem = static_cast<int>(smem);
  }
  const int blocks = cached_blocks;
  lock.unlock();
  set_job_split(P, blocks);
  void *args[] = {&P, const_cast<Exp2Table *>(&tab)};
  return cudaLaunchCooperativeKernel(reinterpret_cast<void *>(pass_kernel<TE>),
                                     dim3(blocks), dim3(kPThreads), args, smem, stream);
}

cudaError_t launch_pass(const Params &P, int esize, const Exp2Table &tab, size_t smem,
                        cudaStream_t stream) {
  return esize == 2 ? launch_pass_t<uint16_t>(P, tab, smem, stream)
                    : launch_pass_t<float>(P, tab, smem, stream);
}

size_t pass_ctl_bytes() { return sizeof(PassCtl); }

}  // namespace sv
