"""Host side of the input recipe for every configuration (no GPU): the seeded
generators and the per-configuration helpers the parity tests and the bench rely
on produce well-formed inputs of the stated shapes."""
import numpy as np
import pytest

from csa2_compressed_sparse_02_gb300 import inputs as I

ALL = list(I.CONFIGS.values()) + [I.PREFILL]


@pytest.mark.parametrize("cfg", ALL, ids=lambda c: "config%d" % c.number)
def test_recipe_helpers_for_every_configuration(cfg):
    lengths = cfg.first_lengths()
    assert len(lengths) == cfg.B and min(lengths) >= 1
    s = 0
    n_c = lengths[s] // cfg.ratio
    pos, rv, rs = I.plants(cfg, 0, s)
    assert pos.size == cfg.plants and (pos.size == 0 or pos.max() < n_c)
    if pos.size:
        assert rv.shape == (I.DI // 2,) and rs.shape == (I.DI // 16,)
    qv, qs, w = I.host_index_q(cfg, 0, s, 0)
    assert qv.shape == (I.HI, I.DI // 2) and qs.shape == (I.HI, I.DI // 16) and w.shape == (I.HI,)
    kv, ks = I.host_index_keys(cfg, 0, s, min(n_c, 4096))
    assert kv.shape == (min(n_c, 4096), I.DI // 2)
    q = I.host_q(cfg, cfg.layer(0, 0), s, 0)
    assert q.shape == (I.H, I.D) and np.isfinite(q).all()
    assert I.host_kv(cfg, 0, s, 0, 3).shape == (3, I.D)


def test_ratio_one_configuration_has_n_c_equal_to_t():
    cfg = I.CONFIGS[7]
    assert cfg.ratio == 1 and cfg.first_lengths()[0] // cfg.ratio == cfg.T
