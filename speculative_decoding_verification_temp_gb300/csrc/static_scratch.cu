// spec_verify_chain_static: spec_verify_chain with its workspace taken from a
// fixed scratch array in this library's device data, so that the call itself
// allocates nothing.  The verification is the same code path: this file only
// checks the arguments, finds the scratch and forwards to spec_verify_chain.
#include <cuda_runtime.h>

#include "specverify.h"

namespace sv {
spec_status check_chain_args(const void *target_logits, int64_t ld_target,
                             const void *draft_logits, int64_t ld_draft, spec_dtype dtype, int B,
                             int gamma, int V, const int32_t *draft_tokens,
                             spec_policy target_policy, spec_policy draft_policy,
                             const int32_t *out_num_accepted, const int32_t *out_tokens);
}  // namespace sv

namespace {

// Static device storage, one copy per device context.  Nothing in it has to
// start at zero: spec_verify_chain clears the part that must (its counters and
// task queue) at the start of every call.
__device__ __align__(256) unsigned char g_scratch[SPEC_STATIC_SCRATCH_BYTES];

// Address of g_scratch in the context current on this thread.  Looked up on
// every call rather than cached: after a device reset (or after the primary
// context was released and created again) the module is loaded anew and an
// address kept from the old context would point at unmapped memory.  Once the
// module is loaded the lookup is a host-side table read.
spec_status scratch_address(void **out) {
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return SPEC_ERR_CUDA;
  *out = p;
  return SPEC_OK;
}

}  // namespace

extern "C" spec_status spec_verify_chain_static(
    const void *target_logits, int64_t ld_target, const void *draft_logits, int64_t ld_draft,
    spec_dtype dtype, int B, int gamma, int V, const int32_t *draft_tokens,
    spec_policy target_policy, spec_policy draft_policy, uint64_t seed,
    const float *uniform_override, int32_t *out_num_accepted, int32_t *out_tokens,
    uint32_t *out_flags, float *out_residual, spec_stream_t stream) {
  // The same argument checks as spec_verify_chain, before the size check, so
  // that a bad argument reads SPEC_ERR_INVALID_ARG here too.
  const spec_status chk = sv::check_chain_args(target_logits, ld_target, draft_logits, ld_draft,
                                               dtype, B, gamma, V, draft_tokens, target_policy,
                                               draft_policy, out_num_accepted, out_tokens);
  if (chk != SPEC_OK || B == 0) return chk;
  // Shapes whose workspace exceeds the scratch are refused before any CUDA call.
  const size_t need = spec_verify_chain_workspace_size(B, gamma, V, dtype);
  if (need == 0 || need > static_cast<size_t>(SPEC_STATIC_SCRATCH_BYTES))
    return SPEC_ERR_UNSUPPORTED;
  void *ws = nullptr;
  const spec_status s = scratch_address(&ws);
  if (s != SPEC_OK) return s;
  return spec_verify_chain(target_logits, ld_target, draft_logits, ld_draft, dtype, B, gamma, V,
                           draft_tokens, target_policy, draft_policy, seed, uniform_override,
                           out_num_accepted, out_tokens, out_flags, out_residual, ws,
                           SPEC_STATIC_SCRATCH_BYTES, stream);
}
