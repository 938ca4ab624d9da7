// The megakernel with every op, for models with MLA and / or MoE layers.
#define MK_VARIANT_FULL 1
#define MK_VARIANT_NS full
#include "mk_kernel.cuh"
