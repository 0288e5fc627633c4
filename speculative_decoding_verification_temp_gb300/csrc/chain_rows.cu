// The rows kernel of the chain path: the pass that reads every logit row of
// the batch from HBM exactly once (see verify_chain.cu for the whole path).
//
// Every logit row of the batch - the gamma + 1 target rows and the gamma draft
// rows of each sequence - is cut into 32 KB chunks, numbered position-major
// (the bonus rows last) and handed out round-robin over a persistent grid
// (three CTAs per SM).  In each
// CTA one producer warp streams its chunks into a ring of two shared-memory
// slots with bulk asynchronous copies (cp.async.bulk, one "full" and one
// "empty" mbarrier per slot); eight consumer warps reduce each chunk to one
// 64-bit record per warp: the (max, sum of 2^((z - max) k)) of a sampling row,
// k = log2(e) / T, or the (finite max, lowest index + 1) of a greedy row.  Each
// logit costs one exponential; nothing else happens on this path (no atomics,
// no cross-CTA waits).  Every mbarrier wait is bounded (about two seconds) and
// sets the error word, which turns into SPEC_FLAG_TIMEOUT.
//
// Trees take the same stream (the tree walk of verify_chain.cu reads the
// records): the N target rows of each tree, then its N draft rows, of which
// those of leaves (no child is ever tested against them) and all of them when
// the target is greedy are skipped.
//
// The same stream serves typical acceptance (kTyp): only the gamma + 1 target
// rows of each sequence, and each warp's record of a sampling row is
// (max, S1 = sum 2^t, S2 = sum 2^t t, lowest index of the max), t = (z - max) k,
// from which the row's entropy and p(x) follow.
#include <mutex>

#include "ops.cuh"

namespace sv {
namespace {

constexpr int kRConsumerWarps = kChainRecordsPerChunk;
constexpr int kRProducerWarp = kRConsumerWarps;
constexpr int kRThreads = (kRConsumerWarps + 1) * 32;  // 288
constexpr int kRMaxRing = 8;
constexpr uint32_t kNoIndex = 0x3FFFFFFFu;  // record index: no finite entry
constexpr uint32_t kBadBit = 0x80000000u;   // record index bit: NaN or +inf seen
static_assert(kRConsumerWarps == 8, "the fast record paths cover 32 KB chunks with 8 warps");

__device__ __forceinline__ void mbar_arrive1_c(unsigned long long *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// What the producer tells the consumers about the chunk in a slot.
struct SlotInfo {
  const void *gl;  // the chunk in global memory
  long long rec;   // index of the chunk's first record
  int n;           // entries
  int nb;          // entries copied to shared memory
  float k;         // log2(e) / T, 0 for a greedy row
  int arg;         // 1: greedy row (argmax record)
  int v0;          // vocabulary index of the chunk's first entry
  int row;         // the chunk's row: seq * (rows per sequence) + r
};

struct RowsCtl {
  unsigned long long full[kRMaxRing];
  unsigned long long empty[kRMaxRing];
  SlotInfo info[kRMaxRing];
};

// Where work item k (a chunk) lives.
struct ChunkInfo {
  int seq, r, c, n;  // sequence, row within the sequence, chunk, entries
  long long row;     // global row of its tensor
  bool draft;
};

// Rows a sequence (or tree) puts on the stream: a chain's gamma + 1 target and
// gamma draft rows, a tree's N target and N draft rows, typical acceptance's
// gamma + 1 target rows.
template <bool kTyp>
__device__ __forceinline__ int stream_rows(const Params &P) {
  return kTyp ? P.gamma + 1 : (P.mode == kModeTree ? 2 * P.ups : 2 * P.gamma + 1);
}

template <bool kTyp>
__device__ __forceinline__ ChunkInfo chunk_info(const Params &P, long long k) {
  ChunkInfo ci;
  const int rps = stream_rows<kTyp>(P);
  const int per_seq = rps * P.cpr;
  const int k32 = static_cast<int>(k);  // the host keeps the chunk count below 2^31
  ci.seq = k32 / per_seq;
  const int rem = k32 - ci.seq * per_seq;
  ci.r = rem / P.cpr;
  ci.c = rem - ci.r * P.cpr;
  ci.n = min(P.chunk_elems, P.V - ci.c * P.chunk_elems);
  if (!kTyp && P.mode == kModeTree) {
    // node-major, from the last node to the root (its draft rows, then its
    // target rows, over every tree): the rows of the shallow nodes, where the
    // walk's passes mostly run, are the last streamed and still in L2 when
    // the walk begins
    const int N = P.ups, T = P.nseq;
    const int g = k32 / P.cpr;  // global row in stream order
    ci.c = k32 - g * P.cpr;
    ci.n = min(P.chunk_elems, P.V - ci.c * P.chunk_elems);
    const int j = g / (2 * T), h = (g / T) & 1;
    ci.seq = g - (g / T) * T;
    const int node = N - 1 - j;
    ci.draft = h == 0;
    ci.r = ci.draft ? N + node : node;
    ci.row = static_cast<long long>(ci.seq) * N + node;
    return ci;
  }
  if (!kTyp) {
    // chains, position-major: the target and draft rows of positions
    // gamma - 1, ..., 1, 0 over every sequence, then the bonus rows.  The rows
    // a draw reads again are most often the bonus row (every draft accepted)
    // and then the pairs of the first positions: streamed last, they are the
    // ones still in L2 when the draw kernel starts.
    const int B = P.nseq, gamma = P.gamma;
    const int g = k32 / P.cpr;  // global row in stream order
    ci.c = k32 - g * P.cpr;
    ci.n = min(P.chunk_elems, P.V - ci.c * P.chunk_elems);
    const int npair = gamma * 2 * B;
    if (g < npair) {
      const int pos = gamma - 1 - g / (2 * B);
      const int h = (g / B) & 1;
      ci.seq = g - (g / B) * B;
      ci.draft = h == 1;
      ci.r = ci.draft ? gamma + 1 + pos : pos;
      ci.row = ci.draft ? static_cast<long long>(ci.seq) * gamma + pos
                        : static_cast<long long>(ci.seq) * (gamma + 1) + pos;
    } else {
      ci.seq = g - npair;
      ci.draft = false;
      ci.r = gamma;
      ci.row = static_cast<long long>(ci.seq) * (gamma + 1) + gamma;
    }
    return ci;
  }
  ci.draft = false;
  ci.row = static_cast<long long>(ci.seq) * (P.gamma + 1) + ci.r;
  return ci;
}

// Policy of a row: greedy (argmax) or sampling with k = log2(e) / T.
__device__ __forceinline__ bool row_is_arg(float T) { return !(T > 0.f) || T == INFINITY; }

// Rows nobody reads are not streamed: the draft rows of a sequence whose
// target is greedy (a one-hot p accepts a draft iff it is p's argmax and needs
// no draw), and the draft rows of a tree's leaves.  The producer decides it;
// such a chunk takes no slot.
template <bool kTyp>
__device__ __forceinline__ bool chunk_skipped(const Params &P, const ChunkInfo &ci) {
  if (kTyp || !ci.draft) return false;
  if (row_is_arg(__ldg(P.Tp + ci.seq))) return true;
  return P.mode == kModeTree && __ldg(P.first_child + ci.row) < 0;
}

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

// Record of this warp's part [e0, e1) of a chunk, any layout: entries below nb
// come from shared memory (groups of 8), the rest (fewer than 8) from global
// memory.
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
  return warp_merge_ms(m, S, k);
}

// Sampling-row record when every group of 8 entries of the warp's part is in
// shared memory: each lane loads all of its groups; the warp takes one max
// (lanes exchange their maxima first, so every lane's terms share the warp's
// scale), then one sum of 2^((z - max) k) over independent packed chains.  A
// NaN propagates into the sum and marks the record bad.
template <typename TE>
__device__ float2 sample_record_fast(const TE *sm, int e0, int e1, float k, TE *bout);

// bout (NULL: none): the maxima of the part's 512-entry blocks go to bout[0..]
// (blocks that start at or past e1 are not written).
template <>
__device__ float2 sample_record_fast<uint16_t>(const uint16_t *sm, int e0, int e1, float k,
                                               uint16_t *bout) {
  const int lane = threadIdx.x & 31;
  constexpr int G = 8;  // 2048 entries per warp
  uint4 w[G];
  if (e0 + G * 256 <= e1) {  // a full part: no per-group bounds
#pragma unroll
    for (int g = 0; g < G; ++g) w[g] = *reinterpret_cast<const uint4 *>(sm + e0 + g * 256 + lane * 8);
  } else {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const int base = e0 + g * 256 + lane * 8;
      w[g] = base < e1 ? *reinterpret_cast<const uint4 *>(sm + base)
                       : make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
    }
  }
  uint32_t h[G];
#pragma unroll
  for (int g = 0; g < G; ++g) h[g] = bf16x2_max(bf16x2_max(w[g].x, w[g].y), bf16x2_max(w[g].z, w[g].w));
  if (bout) {
#pragma unroll
    for (int b = 0; b < G / 2; ++b) {
      uint32_t hb = bf16x2_max(h[2 * b], h[2 * b + 1]);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) hb = bf16x2_max(hb, __shfl_xor_sync(0xFFFFFFFFu, hb, off));
      const uint32_t mb = bf16x2_max(hb, hb >> 16);  // low half: the larger of the two
      if (lane == 0 && e0 + b * 512 < e1) bout[b] = static_cast<uint16_t>(mb & 0xFFFFu);
    }
  }
  uint32_t hh = bf16x2_max(bf16x2_max(bf16x2_max(h[0], h[1]), bf16x2_max(h[2], h[3])),
                           bf16x2_max(bf16x2_max(h[4], h[5]), bf16x2_max(h[6], h[7])));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) hh = bf16x2_max(hh, __shfl_xor_sync(0xFFFFFFFFu, hh, off));
  const float m = fmaxf(__uint_as_float(hh << 16), __uint_as_float(hh & 0xFFFF0000u));
  float S = 0.f;
  if (m == -INFINITY) {  // nothing but -inf and NaN in the whole part: look for NaN
    bool nan = false;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const uint32_t ws[4] = {w[g].x, w[g].y, w[g].z, w[g].w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
        nan |= (ws[i] & 0x7FFFu) > 0x7F80u || (ws[i] & 0x7FFF0000u) > 0x7F800000u;
    }
    S = __any_sync(0xFFFFFFFFu, nan) ? __int_as_float(0x7FC00000) : 0.f;
    return make_float2(m, S);
  }
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
  return make_float2(m, warp_sum(S));  // every lane's terms are relative to the warp's max
}

template <>
__device__ float2 sample_record_fast<float>(const float *sm, int e0, int e1, float k,
                                            float *bout) {
  const int lane = threadIdx.x & 31;
  constexpr int G = 4;  // 1024 entries per warp
  float4 a[G], b[G];
  const float4 ninf = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
  if (e0 + G * 256 <= e1) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      a[g] = *reinterpret_cast<const float4 *>(sm + e0 + g * 256 + lane * 8);
      b[g] = *reinterpret_cast<const float4 *>(sm + e0 + g * 256 + lane * 8 + 4);
    }
  } else {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const int base = e0 + g * 256 + lane * 8;
      a[g] = base < e1 ? *reinterpret_cast<const float4 *>(sm + base) : ninf;
      b[g] = base < e1 ? *reinterpret_cast<const float4 *>(sm + base + 4) : ninf;
    }
  }
  float mg[G];
#pragma unroll
  for (int g = 0; g < G; ++g)
    mg[g] = fmaxf(fmaxf(fmaxf(a[g].x, a[g].y), fmaxf(a[g].z, a[g].w)),
                  fmaxf(fmaxf(b[g].x, b[g].y), fmaxf(b[g].z, b[g].w)));
  if (bout) {
#pragma unroll
    for (int b = 0; b < G / 2; ++b) {
      float mb = fmaxf(mg[2 * b], mg[2 * b + 1]);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, off));
      if (lane == 0 && e0 + b * 512 < e1) bout[b] = mb;
    }
  }
  float m = fmaxf(fmaxf(mg[0], mg[1]), fmaxf(mg[2], mg[3]));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
  float S = 0.f;
  if (m == -INFINITY) {
    bool nan = false;
#pragma unroll
    for (int g = 0; g < G; ++g)
      nan |= a[g].x != a[g].x || a[g].y != a[g].y || a[g].z != a[g].z || a[g].w != a[g].w ||
             b[g].x != b[g].x || b[g].y != b[g].y || b[g].z != b[g].z || b[g].w != b[g].w;
    S = __any_sync(0xFFFFFFFFu, nan) ? __int_as_float(0x7FC00000) : 0.f;
    return make_float2(m, S);
  }
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
  return make_float2(m, warp_sum(S));
}

// Maxima of the warp's 512-entry blocks [e0, e1) of the chunk, stored as the
// element type: bmax[row][block].  Only calls with a row filter ask for them;
// the filter kernel bounds each row's threshold with them.  A lane reads 8
// consecutive entries of each 256-entry half of a block (16-byte loads,
// conflict-free); entries past nb (a chunk whose end is not 16-byte aligned)
// come from global memory.
template <typename TE>
__device__ void block_maxima(const Params &P, const SlotInfo &si, const TE *sm, int e0, int e1) {
  const int lane = threadIdx.x & 31;
  const TE *gl = static_cast<const TE *>(si.gl);
  TE *out = static_cast<TE *>(P.bmax) + static_cast<long long>(si.row) * P.nblk;
  for (int b0 = e0; b0 < e1; b0 += 512) {
    float mx = -INFINITY;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int base = b0 + h * 256 + lane * 8;
      float z[8];
      if (base + 8 <= e1 && base + 8 <= si.nb) {
        load_vec<TE>(sm + base, z);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int e = base + i;
          z[i] = e < e1 ? to_f32(e < si.nb ? sm[e] : gl[e]) : -INFINITY;
        }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) mx = fmaxf(mx, z[i]);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
    if (lane == 0) out[(si.v0 + b0) / 512] = from_f32<TE>(mx);
  }
}

// Typical-acceptance record of this warp's part [e0, e1) of a sampling row's
// chunk: (m, S1, S2, lowest index of m) with m the part's max, t = (z - m) k,
// S1 = sum 2^t, S2 = sum 2^t max(t, -150) (a -inf entry adds 0 to both).  A
// NaN or +inf entry makes S1 NaN (the record is bad).  Entries below nb come
// from shared memory, the rest (fewer than 8) from global memory.
template <typename TE>
__device__ __noinline__ float4 typical_record(const TE *sm, const TE *gl, int e0, int e1, int nb,
                                              int v0, float k) {
  const int lane = threadIdx.x & 31;
  auto group = [&](int base, float z[8]) {
    if (base + 8 <= nb) {
      load_vec<TE>(sm + base, z);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) z[e] = base + e < e1 ? to_f32(gl[base + e]) : -INFINITY;
    }
  };
  float m = -INFINITY;
  for (int base = e0 + lane * 8; base < e1; base += 256) {
    float z[8];
    group(base, z);
#pragma unroll
    for (int e = 0; e < 8; ++e) m = fmaxf(m, z[e]);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
  const uint64_t nm2 = pack2(-m, -m), k2 = pack2(k, k);
  uint64_t s1 = 0ull, s2 = 0ull;
  uint32_t idx = kNoIndex;
  bool nan = false;
  for (int base = e0 + lane * 8; base < e1; base += 256) {
    float z[8];
    group(base, z);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      nan |= z[e] != z[e];
      if (z[e] == m && m > -INFINITY && idx == kNoIndex) idx = static_cast<uint32_t>(v0 + base + e);
    }
    if (m == -INFINITY) continue;
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      const uint64_t t2 = fmul2(fadd2(pack2(z[e], z[e + 1]), nm2), k2);
      const uint64_t w2 = ex2_pair(t2);
      float t0, t1;
      unpack2(t2, t0, t1);
      s1 = fadd2(s1, w2);
      s2 = ffma2(w2, pack2(fmaxf(t0, -150.f), fmaxf(t1, -150.f)), s2);
    }
  }
  float S1 = hsum2(s1), S2 = hsum2(s2);
  S1 = warp_sum(S1);
  S2 = warp_sum(S2);
  nan = __any_sync(0xFFFFFFFFu, nan);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) idx = min(idx, __shfl_xor_sync(0xFFFFFFFFu, idx, off));
  if (nan || m == INFINITY) S1 = __int_as_float(0x7FC00000);
  return make_float4(m, S1, S2, __uint_as_float(idx));
}

// typical_record when the warp's part is entirely in shared memory (entries a
// multiple of 8): one load into registers, packed sums over independent
// chains.  A NaN reaches S1 through the exponential; a -inf entry (whose
// 2^t t would be NaN) sends the part to the clamped path.  The index field is
// left empty: the merge kernel searches the one part that holds the row's max.
template <typename TE>
__device__ float4 typical_record_fast(const TE *sm, int e0, int e1, int v0, float k);

template <>
__device__ float4 typical_record_fast<uint16_t>(const uint16_t *sm, int e0, int e1, int v0,
                                                float k) {
  const int lane = threadIdx.x & 31;
  constexpr int G = 8;  // 2048 entries per warp
  uint4 w[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const int base = e0 + g * 256 + lane * 8;
    w[g] = base < e1 ? *reinterpret_cast<const uint4 *>(sm + base)
                     : make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
  }
  uint32_t hh = 0xFF80FF80u;
#pragma unroll
  for (int g = 0; g < G; ++g)
    hh = bf16x2_max(hh, bf16x2_max(bf16x2_max(w[g].x, w[g].y), bf16x2_max(w[g].z, w[g].w)));
  const float lm = fmaxf(__uint_as_float(hh << 16), __uint_as_float(hh & 0xFFFF0000u));
  float m = lm;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
  if (!(m > -INFINITY) || m == INFINITY) return make_float4(m, __int_as_float(0x7FC00000), 0.f, 0.f);
  const uint64_t nm2 = pack2(-m, -m), k2 = pack2(k, k);
  uint64_t a1[2] = {0ull, 0ull}, a2[2] = {0ull, 0ull};
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const uint32_t ws[4] = {w[g].x, w[g].y, w[g].z, w[g].w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint64_t t2 = fmul2(fadd2(bf16x2_to_pair(ws[q]), nm2), k2);
      const uint64_t e2 = ex2_pair(t2);
      a1[q & 1] = fadd2(a1[q & 1], e2);
      a2[q & 1] = ffma2(e2, t2, a2[q & 1]);
    }
  }
  float S1 = hsum2(fadd2(a1[0], a1[1]));
  float S2 = hsum2(fadd2(a2[0], a2[1]));
  S1 = warp_sum(S1);
  S2 = warp_sum(S2);
  return make_float4(m, S1, S2, __uint_as_float(kNoIndex));  // the merge finds the index
}

template <>
__device__ float4 typical_record_fast<float>(const float *sm, int e0, int e1, int v0, float k) {
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
  float lm = -INFINITY;
#pragma unroll
  for (int g = 0; g < G; ++g)
    lm = fmaxf(lm, fmaxf(fmaxf(fmaxf(a[g].x, a[g].y), fmaxf(a[g].z, a[g].w)),
                         fmaxf(fmaxf(b[g].x, b[g].y), fmaxf(b[g].z, b[g].w))));
  float m = lm;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
  if (!(m > -INFINITY) || m == INFINITY) return make_float4(m, __int_as_float(0x7FC00000), 0.f, 0.f);
  const uint64_t nm2 = pack2(-m, -m), k2 = pack2(k, k);
  uint64_t a1[4] = {0ull, 0ull, 0ull, 0ull}, a2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const uint64_t p[4] = {pack2(a[g].x, a[g].y), pack2(a[g].z, a[g].w), pack2(b[g].x, b[g].y),
                           pack2(b[g].z, b[g].w)};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint64_t t2 = fmul2(fadd2(p[q], nm2), k2);
      const uint64_t e2 = ex2_pair(t2);
      a1[q] = fadd2(a1[q], e2);
      a2[q] = ffma2(e2, t2, a2[q]);
    }
  }
  float S1 = hsum2(fadd2(fadd2(a1[0], a1[1]), fadd2(a1[2], a1[3])));
  float S2 = hsum2(fadd2(fadd2(a2[0], a2[1]), fadd2(a2[2], a2[3])));
  S1 = warp_sum(S1);
  S2 = warp_sum(S2);
  return make_float4(m, S1, S2, __uint_as_float(kNoIndex));  // the merge finds the index
}

template <typename TE, bool kTyp>
__device__ void rows_consumer(const Params &P, RowsCtl &ctl, unsigned char *ring,
                              long long total) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NS = P.ring;
  const int EW = P.chunk_elems / kRConsumerWarps;  // entries per warp (a multiple of 256)
  // the slots the producer fills: this CTA's chunks that are streamed, then
  // an end marker (n < 0); at most one per chunk of this CTA, plus the marker
  const long long cap = (total - blockIdx.x + gridDim.x - 1) / gridDim.x + 1;
  for (long long i = 0; i < cap; ++i) {
    const int slot = static_cast<int>(i % NS);
    const uint32_t phase = static_cast<uint32_t>(i / NS) & 1u;
    if (!mbar_wait_limit(&ctl.full[slot], phase, P.first_wait)) {
      // gave up: flag it, then wait again with the full bound, so that no copy
      // is left in flight and the chunk is read only once it has landed
      if (lane == 0) atomicOr(P.err, 1u);
      mbar_wait_bounded(&ctl.full[slot], phase);
    }
    const SlotInfo si = ctl.info[slot];
    if (si.n < 0) {  // the end marker
      __syncwarp();
      if (lane == 0) mbar_arrive1_c(&ctl.empty[slot]);
      break;
    }
    const TE *sm = reinterpret_cast<const TE *>(ring + static_cast<size_t>(slot) * P.slot_bytes);
    const int e0 = min(si.n, warp * EW), e1 = min(si.n, e0 + EW);
    if (kTyp) {
      float4 rec;
      if (si.arg) {
        const float2 a = chunk_record<TE>(sm, static_cast<const TE *>(si.gl), e0, e1, si.nb,
                                          si.v0, true, 0.f);
        rec = make_float4(a.x, 0.f, 0.f, a.y);
      } else {
        rec = make_float4(0.f, 0.f, 0.f, 0.f);
        const bool fast = si.nb == si.n && (si.n & 7) == 0;
        if (fast) rec = typical_record_fast<TE>(sm, e0, e1, si.v0, si.k);
        // S2 is NaN with S1 finite only when a -inf entry met 2^t t: the
        // clamped path then
        if (!fast || (rec.z != rec.z && rec.y == rec.y) || !(rec.x > -INFINITY))
          rec = typical_record<TE>(sm, static_cast<const TE *>(si.gl), e0, e1, si.nb, si.v0, si.k);
      }
      if (lane == 0) P.trec[si.rec + warp] = rec;  // read by the merge kernel, after this one
      __syncwarp();
      if (lane == 0) mbar_arrive1_c(&ctl.empty[slot]);
      continue;
    }
    const bool fast = !si.arg && si.nb == si.n && (si.n & 7) == 0;
    // the block maxima of a sampled row (calls with a row filter)
    TE *bout = P.bmax && !si.arg ? static_cast<TE *>(P.bmax) +
                                       static_cast<long long>(si.row) * P.nblk + (si.v0 + e0) / 512
                                 : nullptr;
    const float2 rec = fast ? sample_record_fast<TE>(sm, e0, e1, si.k, bout)
                            : chunk_record<TE>(sm, static_cast<const TE *>(si.gl), e0, e1, si.nb,
                                               si.v0, si.arg != 0, si.k);
    if (lane == 0) {
      const unsigned long long bits =
          static_cast<unsigned long long>(__float_as_uint(rec.x)) |
          (static_cast<unsigned long long>(__float_as_uint(rec.y)) << 32);
      P.srec[si.rec + warp] = bits;  // read by the draw kernel, after this kernel
    }
    if (bout && !fast) block_maxima<TE>(P, si, sm, e0, e1);
    __syncwarp();
    if (lane == 0) mbar_arrive1_c(&ctl.empty[slot]);
  }
}

template <typename TE, bool kTyp>
__device__ void rows_producer(const Params &P, RowsCtl &ctl, unsigned char *ring,
                              long long total) {
  const int NS = P.ring;
  const int CE = P.chunk_elems;
  const long long G = gridDim.x;
  // launched behind the first-child kernel (trees): its marks are visible
  // after this wait (a no-op for a launch without programmatic serialisation)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the consumers of the id-th chunk handed its slot back
  auto wait_done = [&](int id) {
    const int slot = id % NS;
    const uint32_t phase = static_cast<uint32_t>(id / NS) & 1u;
    if (!mbar_wait_bounded(&ctl.empty[slot], phase)) atomicOr(P.err, 1u);
  };
  int i = 0;
  for (long long k = blockIdx.x; k < total; k += G) {
    const ChunkInfo ci = chunk_info<kTyp>(P, k);
    if (chunk_skipped<kTyp>(P, ci)) continue;
    const float T = __ldg((ci.draft ? P.Tq : P.Tp) + ci.seq);
    const bool arg = row_is_arg(T);
    const int slot = i % NS;
    if (i >= NS) wait_done(i - NS);
    ++i;
    const TE *gl = static_cast<const TE *>(row_ptr(ci.draft ? P.draft : P.target, ci.row,
                                                   ci.draft ? P.ld_d : P.ld_t, sizeof(TE))) +
                   static_cast<long long>(ci.c) * CE;
    const uint32_t bytes = static_cast<uint32_t>(ci.n * sizeof(TE)) / 16u * 16u;
    SlotInfo &si = ctl.info[slot];
    si.gl = gl;
    const int rps = stream_rows<kTyp>(P);
    si.rec = ((static_cast<long long>(ci.seq) * rps + ci.r) * P.cpr + ci.c) *
             kRConsumerWarps;
    si.n = ci.n;
    si.nb = static_cast<int>(bytes / sizeof(TE));
    si.k = arg ? 0.f : kLog2e / T;
    si.arg = arg ? 1 : 0;
    si.v0 = ci.c * CE;
    si.row = ci.seq * rps + ci.r;
    mbar_arrive_expect_tx(&ctl.full[slot], bytes);
    if (bytes) bulk_g2s_plain(ring + static_cast<size_t>(slot) * P.slot_bytes, gl, bytes,
                              &ctl.full[slot]);
  }
  {  // the end marker: a slot without bytes
    const int slot = i % NS;
    if (i >= NS) wait_done(i - NS);
    ++i;
    ctl.info[slot].n = -1;
    mbar_arrive_expect_tx(&ctl.full[slot], 0u);
  }
  const int issued = i;
  for (int d = max(0, issued - NS); d < issued; ++d) wait_done(d);
}

template <typename TE, bool kTyp>
__global__ void __launch_bounds__(kRThreads, 3) chain_rows_kernel(const Params P) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  RowsCtl &ctl = *reinterpret_cast<RowsCtl *>(smem_raw);
  unsigned char *ring = smem_raw + P.data_off;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long total =
      static_cast<long long>(P.nseq) * stream_rows<kTyp>(P) * static_cast<long long>(P.cpr);
  if (threadIdx.x == 0) {
    for (int s = 0; s < P.ring; ++s) {
      mbar_init(&ctl.full[s], 1);
      mbar_init(&ctl.empty[s], kRConsumerWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();
  if (warp < kRConsumerWarps) {
    rows_consumer<TE, kTyp>(P, ctl, ring, total);
  } else if (warp == kRProducerWarp && lane == 0) {
    rows_producer<TE, kTyp>(P, ctl, ring, total);
  }
  // this CTA's work is done: the next kernel in the stream may start launching
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}


std::mutex g_occ_mu;
int g_occ_dev = -1, g_occ_smem = -1, g_occ_blocks[4] = {0, 0, 0, 0};

template <typename TE, bool kTyp>
cudaError_t launch_rows_t(const Params &P, size_t smem, cudaStream_t stream, bool pdl) {
  auto kern = chain_rows_kernel<TE, kTyp>;
  const int which = (sizeof(TE) == 2 ? 0 : 1) + (kTyp ? 2 : 0);
  int blocks = 0;
  {
    // resident CTAs per SM for the last (device, shared memory) pair, shared
    // by every host thread under the lock
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_occ_mu);
    if (dev != g_occ_dev || static_cast<int>(smem) != g_occ_smem) {
      g_occ_blocks[0] = g_occ_blocks[1] = g_occ_blocks[2] = g_occ_blocks[3] = 0;
      g_occ_dev = dev;
      g_occ_smem = static_cast<int>(smem);
    }
    if (!g_occ_blocks[which]) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem));
      if (e != cudaSuccess) return e;
      int per_sm = 0, sms = 0;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kRThreads, smem);
      if (e != cudaSuccess) return e;
      e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return e;
      if (per_sm < 1) return cudaErrorInvalidConfiguration;
      g_occ_blocks[which] = per_sm * sms;
    }
    blocks = g_occ_blocks[which];
  }
  const long long rps =
      kTyp ? P.gamma + 1 : (P.mode == kModeTree ? 2ll * P.ups : 2ll * P.gamma + 1);
  const long long total = static_cast<long long>(P.nseq) * rps * P.cpr;
  const int grid = static_cast<int>(total < blocks ? total : blocks);
  if (!pdl) {
    kern<<<grid, kRThreads, smem, stream>>>(P);
    return cudaGetLastError();
  }
  // programmatic serialisation: the CTAs may start while the previous kernel
  // drains; only the producer reads what it wrote, after its wait
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kRThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, P);
}

}  // namespace

size_t chain_rows_ctl_bytes() { return sizeof(RowsCtl); }
int chain_records_per_chunk() { return kRConsumerWarps; }

cudaError_t launch_chain_rows(const Params &P, int esize, size_t smem, cudaStream_t stream,
                              bool pdl) {
  return esize == 2 ? launch_rows_t<uint16_t, false>(P, smem, stream, pdl)
                    : launch_rows_t<float, false>(P, smem, stream, pdl);
}

cudaError_t launch_typical_rows(const Params &P, int esize, size_t smem, cudaStream_t stream) {
  return esize == 2 ? launch_rows_t<uint16_t, true>(P, smem, stream, false)
                    : launch_rows_t<float, true>(P, smem, stream, false);
}

}  // namespace sv
