// Sampling walk for dense draft logits with f32 target logits.
#include "walk_sample.cuh"

namespace specv {

cudaError_t launch_walk_sample_logits_f32(const SampleWalkParams &p, cudaStream_t st) {
    if (p.draft_dtype == 1) return launch_ws<0, DRAFT_LOGITS, 1>(p, st);
    return launch_ws<0, DRAFT_LOGITS, 0>(p, st);
}

}  // namespace specv
