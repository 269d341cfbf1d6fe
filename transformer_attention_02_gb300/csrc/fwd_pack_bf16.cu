// Forward-kernel variants in bf16 with the query heads of a K/V group packed into each tile's rows.
#include "attn_fwd_inst.cuh"

ATTN_INSTANTIATE_FWD(/*BF16=*/true, /*ROPE=*/false, /*PACK=*/true)
