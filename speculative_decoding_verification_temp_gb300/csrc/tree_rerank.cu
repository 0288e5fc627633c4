// EAGLE-2 rerank of draft trees: keep the m nodes of highest value.
//
// zzszmyf.github.io "LLM 推测解码精读笔记 · 04 EAGLE：特征空间草稿",
// section 10.3 (扩展 + 重排): value(t_i) is the product of the draft
// confidences c_j along the path from the root to t_i; the rerank keeps the m
// nodes of highest value over the whole tree and flattens them into one
// sequence for verification; ties go to the shallower node.  Because c <= 1 a
// child's value never exceeds its parent's, so the kept set is a connected
// tree (section 题 5).  Remaining ties go to the lower node index.
//
// One CTA of 1024 threads per tree (N <= 4096 nodes, all in shared memory):
//   1. parents and confidences in; confidences clamped into [0, 1] (NaN -> 0,
//      flagged); an invalid parent array (parent[0] != -1 or parent[n] not in
//      [0, n)) ends the tree with nothing kept;
//   2. depths by pointer jumping (about log2 N rounds);
//   3. nodes bucketed by depth (counting sort), then values level by level
//      by one warp, value[n] = value[parent[n]] * c[n] in float32, so every
//      product is taken in the same order as the path from the root;
//   4. one 64-bit key per node, (~value bits, depth, index), ascending in the
//      wanted order, bitonic-sorted; the key of rank m - 1 is the cut;
//   5. kept nodes in ascending index (parents before children) through an
//      exclusive scan, with their parents re-indexed into that list.
#include <climits>

#include "common.cuh"

namespace sv {

namespace {

constexpr int kRrThreads = 1024;
constexpr int kRrWarps = kRrThreads / 32;
constexpr int kRrMaxNodes = 4096;

__device__ __forceinline__ unsigned long long rerank_key(float v, int d, int n) {
  // v in [0, 1]: its bits grow with it, so the complement sorts it descending
  return (static_cast<unsigned long long>(0xFFFFFFFFu - __float_as_uint(v)) << 24) |
         (static_cast<unsigned long long>(d) << 12) | static_cast<unsigned long long>(n);
}

// Exclusive prefix sum of a[0..L) in place (L <= 4 * kRrThreads); returns the
// total.  Each thread owns a run of consecutive entries.
__device__ int block_exclusive_scan(int *a, int L, int *warp_tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int per = (L + kRrThreads - 1) / kRrThreads;
  const int b0 = threadIdx.x * per, b1 = min(L, b0 + per);
  int s = 0;
  for (int i = b0; i < b1; ++i) s += a[i];
  int incl = s;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = warp_tot[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xFFFFFFFFu, w, off);
      if (lane >= off) w += o;
    }
    warp_tot[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  int run = incl - s + (warp > 0 ? warp_tot[warp - 1] : 0);
  for (int i = b0; i < b1; ++i) {
    const int x = a[i];
    a[i] = run;
    run += x;
  }
  const int total = warp_tot[kRrWarps - 1];
  __syncthreads();
  return total;
}

__global__ void __launch_bounds__(kRrThreads) tree_rerank_kernel(
    const int32_t *parent, const float *confidence, int N, int P, int m, int32_t *out_nodes,
    int32_t *out_parent, float *out_value, int32_t *out_count, uint32_t *out_flags) {
  extern __shared__ __align__(16) unsigned char dyn[];
  unsigned long long *keys = reinterpret_cast<unsigned long long *>(dyn);  // [P]
  int *par = reinterpret_cast<int *>(keys + P);  // [N]
  int *dep = par + N;                            // [N]
  int *anc = dep + N;                            // [N]
  float *val = reinterpret_cast<float *>(anc + N);  // [N]
  int *order = reinterpret_cast<int *>(val + N);    // [N] nodes by depth, then positions
  int *lvl = order + N;                             // [N + 1] per-depth counts / offsets
  __shared__ int warp_tot[kRrWarps];
  __shared__ int max_depth;

  const int t = blockIdx.x;
  const long long base = static_cast<long long>(t) * N;
  const long long obase = static_cast<long long>(t) * m;
  constexpr int kPer = kRrMaxNodes / kRrThreads;

  // 1. inputs
  int bad = 0, clamped = 0;
  for (int n = threadIdx.x; n < N; n += kRrThreads) {
    const int p = __ldg(parent + base + n);
    const float c = __ldg(confidence + base + n);
    par[n] = p;
    bad |= n == 0 ? p != -1 : (p < 0 || p >= n);
    clamped |= !(c >= 0.f && c <= 1.f);
    val[n] = c > 0.f ? fminf(c, 1.f) : 0.f;
  }
  bad = __syncthreads_or(bad);
  clamped = __syncthreads_or(clamped);
  if (bad) {
    for (int i = threadIdx.x; i < m; i += kRrThreads) {
      out_nodes[obase + i] = -1;
      out_parent[obase + i] = -1;
      if (out_value) out_value[obase + i] = 0.f;
    }
    if (threadIdx.x == 0) {
      out_count[t] = 0;
      if (out_flags) out_flags[t] = SPEC_FLAG_BAD_TREE;
    }
    return;
  }

  // 2. depths: anc[n] jumps towards the root, dep[n] counts the links passed
  for (int n = threadIdx.x; n < N; n += kRrThreads) {
    anc[n] = par[n];
    dep[n] = n == 0 ? 0 : 1;
  }
  if (threadIdx.x == 0) max_depth = 0;
  __syncthreads();
  for (int span = 1; span < N; span <<= 1) {
    int na[kPer], nd[kPer];
#pragma unroll
    for (int r = 0; r < kPer; ++r) {
      const int n = threadIdx.x + r * kRrThreads;
      if (n < N) {
        const int a = anc[n];
        na[r] = a >= 0 ? anc[a] : -1;
        nd[r] = a >= 0 ? dep[n] + dep[a] : dep[n];
      }
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kPer; ++r) {
      const int n = threadIdx.x + r * kRrThreads;
      if (n < N) {
        anc[n] = na[r];
        dep[n] = nd[r];
      }
    }
    __syncthreads();
  }

  // 3. bucket by depth, then values from the root down
  for (int d = threadIdx.x; d <= N; d += kRrThreads) lvl[d] = 0;
  __syncthreads();
  for (int n = threadIdx.x; n < N; n += kRrThreads) {
    atomicAdd(&lvl[dep[n]], 1);
    atomicMax(&max_depth, dep[n]);
  }
  __syncthreads();
  const int D = max_depth;
  block_exclusive_scan(lvl, D + 1, warp_tot);
  for (int n = threadIdx.x; n < N; n += kRrThreads) order[atomicAdd(&lvl[dep[n]], 1)] = n;
  __syncthreads();  // lvl[d] is now the end of level d
  // one warp walks the levels (a level holds a few nodes in a draft tree, so
  // a warp barrier per level beats a block barrier)
  if (threadIdx.x < 32) {
    for (int d = 1; d <= D; ++d) {
      const int b = lvl[d - 1], e = lvl[d];
      for (int i = b + static_cast<int>(threadIdx.x); i < e; i += 32) {
        const int n = order[i];
        val[n] = __fmul_rn(val[par[n]], val[n]);
      }
      __syncwarp();
    }
  }
  __syncthreads();

  // 4. keys, bitonic sort, the cut
  for (int i = threadIdx.x; i < P; i += kRrThreads)
    keys[i] = i < N ? rerank_key(val[i], dep[i], i) : ~0ull;
  __syncthreads();
  for (int k = 2; k <= P; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < P; i += kRrThreads) {
        const int l = i ^ j;
        if (l > i) {
          const unsigned long long a = keys[i], b = keys[l];
          if ((a > b) == ((i & k) == 0)) {
            keys[i] = b;
            keys[l] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  const int count = min(m, N);
  const unsigned long long cut = keys[count - 1];

  // 5. kept nodes in index order, parents re-indexed
  for (int n = threadIdx.x; n < N; n += kRrThreads)
    order[n] = rerank_key(val[n], dep[n], n) <= cut ? 1 : 0;
  __syncthreads();
  block_exclusive_scan(order, N, warp_tot);
  for (int n = threadIdx.x; n < N; n += kRrThreads) {
    if (rerank_key(val[n], dep[n], n) > cut) continue;
    const int p = order[n];
    out_nodes[obase + p] = n;
    out_parent[obase + p] = n == 0 ? -1 : order[par[n]];
    if (out_value) out_value[obase + p] = val[n];
  }
  for (int i = count + threadIdx.x; i < m; i += kRrThreads) {
    out_nodes[obase + i] = -1;
    out_parent[obase + i] = -1;
    if (out_value) out_value[obase + i] = 0.f;
  }
  if (threadIdx.x == 0) {
    out_count[t] = count;
    if (out_flags) out_flags[t] = clamped ? SPEC_FLAG_NONFINITE : 0u;
  }
}

}  // namespace

cudaError_t launch_tree_rerank(const int32_t *parent, const float *confidence, int T, int N, int m,
                               int32_t *out_nodes, int32_t *out_parent, float *out_value,
                               int32_t *out_count, uint32_t *out_flags, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  if (N < 1 || N > kRrMaxNodes || m < 1) return cudaErrorInvalidValue;
  int P = 1;
  while (P < N) P <<= 1;
  const size_t smem = static_cast<size_t>(P) * sizeof(unsigned long long) +
                      static_cast<size_t>(N) * (5 * sizeof(int) + sizeof(float)) + sizeof(int);
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(
        tree_rerank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  tree_rerank_kernel<<<T, kRrThreads, smem, stream>>>(parent, confidence, N, P, m, out_nodes,
                                                      out_parent, out_value, out_count, out_flags);
  return cudaGetLastError();
}

}  // namespace sv
