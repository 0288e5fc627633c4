// Ancestor-or-self tree masks and depth position ids.
//
// whoami-wesleyyou.top "Speculative Decoding" notes, section "Token Tree
// Verifier: topology-aware causal mask": a flattened candidate tree needs a
// mask under which every node sees the shared prefix, its own ancestors and
// itself, and never a sibling branch; positions follow the depth along the
// path.  jennyma11.github.io "11.3 Self-Draft", section 11.3.4 Tree Attention:
// position ids by path depth, not by flattened index.
//
// One CTA per tree: the parent array is staged in shared memory, one warp
// builds one node's mask row (each lane owns words lane and lane + 32 of the
// row, so a row of up to 64 words is written with two coalesced stores) by
// walking the node's parent chain.  Cost is O(N * depth) shared-memory reads
// per tree.
#include "common.cuh"

namespace sv {

__global__ void __launch_bounds__(kThreads)
    tree_mask_kernel(const int32_t *parent, int N, int max_depth, uint64_t *mask,
                     int32_t *position, uint32_t *flags) {
  extern __shared__ int par_s[];
  __shared__ uint32_t red[kWarps];
  const int t = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long long base = static_cast<long long>(t) * N;
  for (int n = threadIdx.x; n < N; n += kThreads) par_s[n] = __ldg(parent + base + n);
  __syncthreads();
  const int words = (N + 63) / 64;
  uint32_t tf = 0u;
  if (threadIdx.x == 0 && par_s[0] != -1) tf |= SPEC_FLAG_BAD_TREE;
  for (int n = warp; n < N; n += kWarps) {
    unsigned long long w0 = 0ull, w1 = 0ull;
    int a = n, d = 0;
    bool ok = true;
    for (;;) {
      const int word = a >> 6;
      const unsigned long long bit = 1ull << (a & 63);
      if (word == lane) w0 |= bit;
      if (word == lane + 32) w1 |= bit;
      if (a == 0) break;
      const int pa = par_s[a];
      if (!(pa >= 0 && pa < a)) {
        ok = false;
        break;
      }
      a = pa;
      ++d;
    }
    uint64_t *row = mask + (base + n) * words;
    if (lane < words) row[lane] = w0;
    if (lane + 32 < words) row[lane + 32] = w1;
    if (lane == 0) {
      position[base + n] = ok ? d : -1;
      if (!ok) tf |= SPEC_FLAG_BAD_TREE;
      if (ok && d > max_depth) tf |= SPEC_FLAG_DEPTH;
    }
  }
  tf = warp_or(tf);
  if (lane == 0) red[warp] = tf;
  __syncthreads();
  if (threadIdx.x == 0 && flags) {
    uint32_t f = 0u;
    for (int w = 0; w < kWarps; ++w) f |= red[w];
    flags[t] = f;
  }
}

cudaError_t launch_tree_mask(const int32_t *parent, int T, int N, int max_depth, uint64_t *mask,
                             int32_t *position, uint32_t *flags, cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(N) * sizeof(int);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(tree_mask_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  tree_mask_kernel<<<T, kThreads, smem, stream>>>(parent, N, max_depth, mask, position, flags);
  return cudaGetLastError();
}

}  // namespace sv
