"""The seeded input generators (workloads/): the recipe the design notes state —
distinct routed ids per token, the shared expert last with weight 1.0, softmax
router weights, scale bytes in [118, 124], N(0, 1) hidden states, Zipf skew with
expert 0 hottest — and determinism per seed.  Small d_model / d_inter keep the
weight tensors cheap; the routing draws are those of the full workloads."""
import numpy as np
import pytest
import torch

import workloads


def _small(T, E, K, zipf=None):
    return workloads.custom(T, 128, 128, E, K, zipf=zipf)


@pytest.mark.parametrize("T,E,K,zipf", [(16, 9, 3, None), (128, 257, 9, None), (512, 33, 9, None),
                                        (4096, 257, 9, 1.2)])
def test_routing_recipe(T, E, K, zipf):
    inp = workloads.make_inputs(_small(T, E, K, zipf), seed=0)
    ids = inp["topk_ids"].numpy()
    wts = inp["topk_weights"].numpy()
    assert ids.shape == (T, K) and ids.dtype == np.int32 and wts.dtype == np.float32
    assert (ids[:, -1] == E - 1).all() and (wts[:, -1] == 1.0).all()
    routed = ids[:, :-1]
    assert ((routed >= 0) & (routed < E - 1)).all()
    assert all(len(set(row)) == K - 1 for row in routed.tolist())
    rw = wts[:, :-1]
    assert (rw > 0).all()
    np.testing.assert_allclose(rw.sum(axis=1), 1.0, atol=1e-5)


def test_uniform_and_zipf_expert_loads():
    uni = workloads.make_inputs(_small(4096, 257, 9), seed=0)["topk_ids"].numpy()[:, :-1]
    cu = np.bincount(uni.reshape(-1), minlength=256)
    assert cu.min() > 0 and cu.max() < 2 * cu.min()          # about 144 each
    zpf = workloads.make_inputs(_small(4096, 257, 9, 1.2), seed=0)["topk_ids"].numpy()[:, :-1]
    cz = np.bincount(zpf.reshape(-1), minlength=256)
    assert cz.argmax() == 0 and cz[0] > 0.9 * 4096           # nearly every token hits expert 0
    assert (cz > 0).all()                                   # every routed expert is touched
    assert cz[:8].sum() > cz[128:].sum()                    # the head outweighs the tail


def test_value_distributions():
    inp = workloads.make_inputs(_small(64, 9, 3), seed=0)
    h = inp["hidden"].float().numpy()
    assert abs(h.mean()) < 0.05 and abs(h.std() - 1.0) < 0.05
    for k in ("w13_scale", "w2_scale"):
        s = inp[k].numpy()
        assert s.min() == 118 and s.max() == 124
    for k in ("w13", "w2"):
        c = inp[k].numpy()
        assert c.min() == 0 and c.max() == 255


def test_seeded_and_deterministic():
    w = _small(32, 17, 5)
    a = workloads.make_inputs(w, seed=3)
    b = workloads.make_inputs(w, seed=3)
    c = workloads.make_inputs(w, seed=4)
    for k in a:
        assert torch.equal(a[k], b[k]), k
    assert not torch.equal(a["hidden"], c["hidden"])
    assert not torch.equal(a["topk_ids"], c["topk_ids"])
