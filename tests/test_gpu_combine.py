"""GPU parity of qattn_combine (log-sum-exp merge) against the oracle."""

import numpy as np
import pytest
import torch

from common import assert_close_lse, require_gpu
from oracle import attention as att

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("S,R,D", [(1, 5, 128), (7, 33, 64), (256, 64, 128), (1024, 3, 128)])
def test_combine(S, R, D):
    qa = require_gpu()
    rng = np.random.default_rng(S * 1000 + R)
    po = rng.standard_normal((S, R, D)).astype(np.float32)
    pl = (rng.standard_normal((S, R)) * 5).astype(np.float32)
    pl[rng.random((S, R)) < 0.2] = -np.inf           # empty splits
    pl[:, 0] = -np.inf                                # a row whose every split is empty
    po[np.isneginf(pl)] = np.nan                      # never read
    out, lse = qa.combine(torch.from_numpy(po).cuda(), torch.from_numpy(pl).cuda(), return_lse=True)
    O, L = att.combine(np.nan_to_num(po), pl)
    o = out.float().cpu().numpy()
    assert np.isfinite(o).all()
    # fp16 output: half an ulp of |O| plus fp32 accumulation
    assert (np.abs(o - O) <= np.abs(O) * 2.0**-11 + 1e-5).all()
    assert_close_lse(lse, L, tol=1e-5)
