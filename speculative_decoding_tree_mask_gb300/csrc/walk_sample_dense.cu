// Sampling walk for dense drafts: draft probabilities here; draft logits by target dtype in
// walk_sample_logits_bf16.cu and walk_sample_logits_f32.cu (separate units compile in
// parallel).
#include "walk_sample.cuh"

namespace specv {

cudaError_t launch_walk_sample_logits_bf16(const SampleWalkParams &p, cudaStream_t st);
cudaError_t launch_walk_sample_logits_f32(const SampleWalkParams &p, cudaStream_t st);

cudaError_t launch_walk_sample_dense(const SampleWalkParams &p, cudaStream_t st) {
    if (p.draft_kind == DRAFT_PROBS_F32) {
        if (p.dtype == 1) return launch_ws<1, DRAFT_PROBS_F32, 0>(p, st);
        return launch_ws<0, DRAFT_PROBS_F32, 0>(p, st);
    }
    if (p.dtype == 1) return launch_walk_sample_logits_bf16(p, st);
    return launch_walk_sample_logits_f32(p, st);
}

}  // namespace specv
