"""The device RoPE table against the oracle's float64 angles."""
import numpy as np
import pytest

import oracle.linattn as ol

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("grid,split", [((25, 22, 40), (44, 42, 42)),
                                        ((181, 22, 40), (44, 42, 42)),
                                        ((3, 5, 7), (8, 6, 114)),
                                        ((2, 1, 1), (128, 0, 0))])
def test_table_matches_oracle_angles(grid, split, cuda_device):
    from gated_linear_attention_attn_b300 import sla
    rt = sla.RopeTable(grid, split, 10000.0, device=cuda_device)
    spec = ol.RopeSpec(*grid, *split, base=10000.0)
    ang = ol.rope3d_angles(spec)                              # [N, 64] float64
    t, h, w = ol.rope3d_positions(spec)
    tt, th, tw = (x.double().cpu().numpy() for x in rt.axis_tables())
    cs = np.concatenate([tt[t], th[h], tw[w]], axis=1)        # [N, 64, 2]
    assert cs.shape == ang.shape + (2,)
    assert np.max(np.abs(cs[..., 0] - np.cos(ang))) <= 1e-6
    assert np.max(np.abs(cs[..., 1] - np.sin(ang))) <= 1e-6
    # the per-token fp16 rows: every pair of every token, rounded to fp16
    tok = rt.token_rows().double().cpu().numpy()              # [N, 64, 2]
    assert tok.shape == ang.shape + (2,)
    assert np.max(np.abs(tok[..., 0] - np.cos(ang))) <= 2.5e-4
    assert np.max(np.abs(tok[..., 1] - np.sin(ang))) <= 2.5e-4
