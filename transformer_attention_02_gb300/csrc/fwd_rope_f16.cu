// Forward-kernel variants in fp16, queries rotated (rotary position embedding) at tile load.
#include "attn_fwd_inst.cuh"

ATTN_INSTANTIATE_FWD(/*BF16=*/false, /*ROPE=*/true, /*PACK=*/false)
