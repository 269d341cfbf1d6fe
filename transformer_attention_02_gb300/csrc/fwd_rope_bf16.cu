// Forward-kernel variants in bf16, queries rotated (rotary position embedding) at tile load.
#include "attn_fwd_inst.cuh"

ATTN_INSTANTIATE_FWD(/*BF16=*/true, /*ROPE=*/true, /*PACK=*/false)
