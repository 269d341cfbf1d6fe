"""GPU parity on a fixed-seed random sweep of shapes, against the FP64 oracle.

Each case draws independently:
- batch and head counts, including GQA ratios that are not powers of two (no head packing) and
  ratios that are (packing when Sq * G fits a tile);
- ragged query and key lengths, with Sq != Sk in both directions;
- the head dimension, the mask kind, and the 16-bit type;
- the entry point: the plain call, or the split-key call with an automatic or a fixed range count.

Every output element of every case is compared, so the sweep crosses combinations that the
hand-picked cases elsewhere take one at a time.
"""
import random

import pytest
import torch

from gpu_helpers import check, run_gpu
from transformer_attention_02_gb300 import attention_splitkv
from transformer_attention_02_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _cases(n=24, seed=20261202):
    rnd = random.Random(seed)
    out = []
    for i in range(n):
        hkv = rnd.choice([1, 2, 4])
        g = rnd.choice([1, 2, 3, 4, 8])
        sq = rnd.choice([1, 2, 7, 64, 129, 200, rnd.randint(1, 400)])
        sk = rnd.choice([sq, rnd.randint(1, 400), 128, 257])
        out.append(dict(
            B=rnd.choice([1, 2, 3]), Hq=hkv * g, Hkv=hkv, Sq=sq, Sk=sk,
            D=rnd.choice([64, 128]), kind=rnd.randrange(4),
            dtype=rnd.choice(["bf16", "f16"]),
            path=rnd.choice(["plain", "plain", "split0", "split3"]),
            seed=1000 + i))
    return out


CASES = _cases()


@pytest.mark.parametrize("c", CASES, ids=lambda c: "B{B}_H{Hq}-{Hkv}_S{Sq}-{Sk}_D{D}_m{kind}_{dtype}_{path}".format(**c))
def test_random_case_matches_oracle(c):
    cfg = I.AttnConfig("sweep", c["B"], c["Hq"], c["Hkv"], c["Sq"], c["Sk"], c["D"],
                       causal=bool(c["kind"] & 1), additive_mask=bool(c["kind"] & 2),
                       seed=c["seed"], dtype=c["dtype"])
    q, k, v, mask = I.make_inputs(cfg)
    if c["path"] == "plain":
        o, lse = run_gpu(q, k, v, mask, cfg.causal)
    else:
        dev = torch.device("cuda")
        o, lse = attention_splitkv(q.to(dev), k.to(dev), v.to(dev), causal=cfg.causal,
                                   mask=None if mask is None else mask.to(dev),
                                   num_splits=0 if c["path"] == "split0" else 3)
        torch.cuda.synchronize()
    check(o, lse, q, k, v, mask, cfg.mask_kind, label=str(c))
