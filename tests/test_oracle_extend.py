"""Pins of the oracle's short causal extend (CPU only).

"Introspective Diffusion Language Model", "3.3 I-DLM Serving Stack": the new
query tokens of a step attend the cached prefix and each other causally.
Pinned against PyTorch SDPA in fp64 (causal attention over the whole
sequence, whose last n rows are exactly the extend), the single-token case
(plain attention over every key) and the causal invariant (a token's output
does not depend on the tokens after it).
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle


def _rand(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float64)


def _sdpa(q, k, v, **kw):
    G = q.shape[1] // k.shape[1]
    qh = q.transpose(0, 1)
    kh = k.repeat_interleave(G, dim=1).transpose(0, 1)
    vh = v.repeat_interleave(G, dim=1).transpose(0, 1)
    return F.scaled_dot_product_attention(qh, kh, vh, **kw).transpose(0, 1)


def _case(P, n, Hq=6, Hkv=2, d=16, seed=0):
    T = P + n
    q = _rand((T, Hq, d), seed)
    k = _rand((T, Hkv, d), seed + 1)
    v = _rand((T, Hkv, d), seed + 2)
    return q, k, v


@pytest.mark.parametrize("P,n", [(0, 1), (0, 5), (7, 3), (37, 9), (130, 4), (5, 1)])
def test_extend_is_the_tail_of_causal_attention(P, n):
    q, k, v = _case(P, n, seed=P + n)
    ref = _sdpa(q, k, v, is_causal=True).numpy()[P:]
    got = oracle.extend(q[P:][None], k[P:][None], v[P:][None], [k[:P]], [v[:P]])[0]
    assert np.abs(got - ref).max() < 1e-12


@pytest.mark.parametrize("P", [1, 16, 100])
def test_single_new_token_sees_every_key(P):
    q, k, v = _case(P, 1, Hq=4, Hkv=4, d=8, seed=3)
    ref = _sdpa(q[P:], k, v).numpy()
    got = oracle.extend(q[P:][None], k[P:][None], v[P:][None], [k[:P]], [v[:P]])[0]
    assert np.abs(got - ref).max() < 1e-12


def test_later_tokens_do_not_change_earlier_outputs():
    P, n = 21, 6
    q, k, v = _case(P, n, seed=11)
    a = oracle.extend(q[P:][None], k[P:][None], v[P:][None], [k[:P]], [v[:P]])[0]
    k2, v2 = k.clone(), v.clone()
    k2[P + 3:] += 5.0
    v2[P + 3:] -= 7.0
    b = oracle.extend(q[P:][None], k2[P:][None], v2[P:][None], [k2[:P]], [v2[:P]])[0]
    assert np.array_equal(a[:3], b[:3])
    assert np.abs(a[3:] - b[3:]).max() > 1e-3


def test_batch_rows_are_independent():
    q0, k0, v0 = _case(9, 4, seed=1)
    q1, k1, v1 = _case(30, 4, seed=2)
    both = oracle.extend(torch.stack([q0[9:], q1[30:]]), torch.stack([k0[9:], k1[30:]]),
                         torch.stack([v0[9:], v1[30:]]), [k0[:9], k1[:30]], [v0[:9], v1[:30]])
    one = oracle.extend(q1[30:][None], k1[30:][None], v1[30:][None], [k1[:30]], [v1[:30]])
    assert np.array_equal(both[1], one[0])
