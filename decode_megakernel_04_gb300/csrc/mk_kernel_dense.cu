// The megakernel for models without MLA or MoE layers (GQA, gated delta net, KDA, dense SwiGLU), plus the
// set-up helper kernels.
#define MK_VARIANT_FULL 0
#define MK_VARIANT_NS dense
#include "mk_kernel.cuh"
