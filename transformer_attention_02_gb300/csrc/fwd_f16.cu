// Forward-kernel variants in fp16, queries used as given.
#include "attn_fwd_inst.cuh"

ATTN_INSTANTIATE_FWD(/*BF16=*/false, /*ROPE=*/false, /*PACK=*/false)
