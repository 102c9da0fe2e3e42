// Sampling walk for point-mass drafts (deterministic tries) and the dispatch of all kinds.
#include "walk_sample.cuh"

namespace specv {

cudaError_t launch_walk_sample_dense(const SampleWalkParams &p, cudaStream_t st);

cudaError_t launch_walk_sample(const SampleWalkParams &p, cudaStream_t st) {
    if (p.B <= 0) return cudaSuccess;
    if (p.draft_kind != DRAFT_POINT) return launch_walk_sample_dense(p, st);
    if (p.dtype == 1) return launch_ws<1, DRAFT_POINT, 0>(p, st);
    return launch_ws<0, DRAFT_POINT, 0>(p, st);
}

}  // namespace specv
