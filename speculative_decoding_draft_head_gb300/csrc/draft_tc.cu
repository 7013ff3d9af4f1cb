// Draft sampling on the tcgen05 tensor cores (bf16 Markov bias); see below.
#include "internal.h"

namespace dspark {

cudaError_t launch_draft_tensor(const DraftArgs &, const DraftPlan &, int, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace dspark
