// MLA latent-cache decode (placeholder until the tensor-core kernel lands).
#include "kvarn_common.cuh"
#include "kvarn_launch.h"

namespace kvarn {

SplitPlan plan_mla(int32_t num_seqs, int32_t max_seq_len) {
  SplitPlan p{};
  p.tiles_per_split = 1;
  p.nsplit = max_seq_len / 128;
  p.slots = p.nsplit + 1;
  (void)num_seqs;
  return p;
}

int64_t mla_workspace_bytes(int32_t num_seqs, int32_t num_heads, const SplitPlan& plan) {
  return static_cast<int64_t>(num_seqs) * num_heads * plan.slots * (512 + 4) * 4;
}

cudaError_t launch_decode_mla(const DecodeParams&, const SplitPlan&, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace kvarn
