// Forward-kernel variants in bf16, queries used as given.
#include "attn_fwd_inst.cuh"

ATTN_INSTANTIATE_FWD(/*BF16=*/true, /*ROPE=*/false, /*PACK=*/false)
