"""Token-tile sizes at the grouped GEMMs' geometry boundaries, against the oracle.

Both GEMMs size a launch's token stages and accumulators from its largest
token tile, and load a tile of n rows (rounded up to 16) in one to three TMA
boxes of 16, 32, 64 or 128 rows.  The W4A16 GEMM adds a 96-row box, keeps one
decoded weight slot at 65-96 rows, and runs every tile of a launch whose largest
tile exceeds 96 rows as two items of up to 64 rows.  Here the routing is built
so that the experts receive exactly the counts at those boundaries; each case
is compared with the oracle (final output within the relative L2 bound of
1e-2), and a few tokens run alone must give their rows of the large batch bit
for bit, so tiles of every size accumulate in the same order
(Megatron-LM PR #8262, "What is tested": batch invariance; FlashInfer PR #5019,
"Tensor and numerical contract").
"""
import numpy as np
import pytest
import torch

import nvfp4_token_routed_gb300 as M
from nvfp4_token_routed_gb300 import workloads as W

from helpers import OracleRun, bf16_np, rel_l2, to_np_u16

pytestmark = pytest.mark.gpu
DEV = "cuda"
E, H, I = 8, 512, 256


def _case(counts, act, seed):
    """Inputs whose top-1 routing gives expert e exactly counts[e] tokens, in a
    shuffled token order."""
    T = int(sum(counts))
    wl = W.Workload(f"tiles_{act}_T{T}_H{H}_I{I}_E{E}_K1", T, H, I, E, 1, act)
    w1, w2 = W.make_weights(wl)
    x = W.make_x(wl)
    g = torch.Generator().manual_seed(W.BASE_SEED + seed)
    ids = torch.repeat_interleave(torch.arange(E, dtype=torch.int32),
                                  torch.tensor(counts, dtype=torch.int64))
    ids = ids[torch.randperm(T, generator=g)].reshape(T, 1).contiguous()
    wts = torch.ones(T, 1, dtype=torch.float32)
    return wl, w1, w2, x, ids, wts


def _alone_rows(run, x, ids, wts, full, seed):
    """Five tokens run as their own batch give their rows of the full batch."""
    g = torch.Generator().manual_seed(W.BASE_SEED + seed)
    sel = torch.randperm(x.shape[0], generator=g)[:5]
    out = run(x[sel].contiguous(), ids[sel].contiguous(), wts[sel].contiguous())
    assert torch.equal(out.view(torch.int16), full[sel.to(DEV)].view(torch.int16))


# W4A16: largest tile 96 (one item per tile, the 96-row box) and above 96 (every
# tile as two items); W4A4: box compositions of 1-3 copies, a multi-tile expert,
# an empty expert, and the one-launch path (at most 8 routes per expert).
W4A16_COUNTS = {
    "max96": [1, 15, 16, 17, 64, 65, 95, 96],
    "max160": [97, 128, 129, 160, 33, 64, 65, 1],
}
W4A4_COUNTS = {
    "boxes": [1, 16, 17, 48, 112, 127, 128, 129],
    "multi_tile_and_empty": [257, 0, 80, 3, 32, 33, 96, 250],
    "one_launch": [1, 2, 15, 16, 17, 0, 13, 0],
}


@pytest.mark.parametrize("act", ["swiglu", "relu2"])
@pytest.mark.parametrize("case", sorted(W4A16_COUNTS))
def test_w4a16_tile_sizes(case, act):
    wl, w1, w2, x, ids, wts = _case(W4A16_COUNTS[case], act, 31)
    w = M.prepare_weights(w1.to(DEV), w2.to(DEV), act)
    xd, idd, wd = x.to(DEV), ids.to(DEV), wts.to(DEV)
    out = M.forward_w4a16(w, xd, idd, wd)
    torch.cuda.synchronize()
    ref = OracleRun(wl, x, w1, w2, ids, wts, w4a16=True)
    got = bf16_np(to_np_u16(out.cpu()))
    want = bf16_np(ref.res["out"])
    assert np.isfinite(got).all()
    assert rel_l2(got, want) <= 1e-2
    _alone_rows(lambda a, b, c: M.forward_w4a16(w, a, b, c), xd, idd, wd, out, 32)


@pytest.mark.parametrize("case", sorted(W4A4_COUNTS))
def test_w4a4_tile_sizes(case):
    wl, w1, w2, x, ids, wts = _case(W4A4_COUNTS[case], "swiglu", 33)
    w = M.prepare_weights(w1.to(DEV), w2.to(DEV), "swiglu")
    xd, idd, wd = x.to(DEV), ids.to(DEV), wts.to(DEV)

    def run(a, b, c):
        codes, sf, scale = M.quantize_tokens(a)
        return M.forward(w, codes, sf, scale, b, c)

    out = run(xd, idd, wd)
    torch.cuda.synchronize()
    ref = OracleRun(wl, x, w1, w2, ids, wts)
    got = bf16_np(to_np_u16(out.cpu()))
    want = bf16_np(ref.res["out"])
    assert np.isfinite(got).all()
    assert rel_l2(got, want) <= 1e-2
    _alone_rows(run, xd, idd, wd, out, 34)
