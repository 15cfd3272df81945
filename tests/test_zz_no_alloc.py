"""The allocation-free Top-K entry point (csa2_topk_static).

Some callers of this library cannot allocate device memory: a plugin whose
host engine owns every device allocation and passes it only inputs and
outputs, or a serving loop that cannot afford cudaMalloc's device-wide
synchronisation. csa2_topk_static serves them with a fixed scratch buffer
inside the library. This file checks, through the C ABI, that it returns
exactly what the workspace-taking csa2_topk returns, on two calls in a row
(the shared buffer keeps the previous call's contents, so the second call
also checks that the call clears what must start at zero), and that a
problem larger than the buffer is refused with its own status code.
"""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa2():
    from fp4_kv_cache_02_gb300 import csa2 as m
    return m


def _run_both(csa2, s, k, n_valid=None, positions=None):
    B, n = s.shape
    ref = torch.empty(B, k, dtype=torch.int32, device="cuda")
    csa2.csa2_topk(s, k, ref, csa2.topk_workspace(B, n, k), n_valid=n_valid, positions=positions)
    got = torch.full((B, k), 7, dtype=torch.int32, device="cuda")
    csa2.csa2_topk_static(s, k, got, n_valid=n_valid, positions=positions)
    torch.cuda.synchronize()
    return ref, got


def test_static_topk_matches_workspace_topk_on_two_calls_in_a_row(csa2):
    g = torch.Generator(device="cuda")
    g.manual_seed(77)
    # call 1: the bench-shaped case, 32 rows of 65,536 scores, k = 512
    s1 = torch.randn(32, 65536, generator=g, device="cuda")
    nv1 = torch.full((32,), 65536, dtype=torch.int32, device="cuda")
    nv1[3] = 1000
    ref, got = _run_both(csa2, s1, 512, n_valid=nv1)
    assert torch.equal(ref, got)
    # call 2: different shape, heavy ties and a positions map, right after call 1
    s2 = torch.randint(0, 4, (3, 20000), generator=g, device="cuda").float()
    pos = torch.randperm(1 << 20, generator=g, device="cuda")[:60000].reshape(3, 20000).to(torch.int32)
    ref, got = _run_both(csa2, s2, 2048, positions=pos)
    assert torch.equal(ref, got)
    assert csa2.csa2_get_last_error() == 0


def test_static_topk_refuses_problems_larger_than_its_buffer(csa2):
    s = torch.zeros(8, 1 << 20, device="cuda")
    idx = torch.empty(8, 512, dtype=torch.int32, device="cuda")
    need = csa2.lib().csa2_topk_workspace_size(8, 1 << 20, 512)
    assert need > csa2.TOPK_STATIC_SCRATCH_BYTES
    with pytest.raises(csa2.Csa2Error) as e:
        csa2.csa2_topk_static(s, 512, idx)
    assert e.value.status == -8


def test_static_topk_limit_is_the_workspace_size(csa2):
    # the largest batch of 65,536-score rows whose csa2_topk workspace fits the
    # buffer is accepted and equals csa2_topk; one more row is refused
    n, k = 65536, 512
    size = csa2.lib().csa2_topk_workspace_size
    B = 1
    while size(B + 1, n, k) <= csa2.TOPK_STATIC_SCRATCH_BYTES:
        B += 1
    assert size(B, n, k) <= csa2.TOPK_STATIC_SCRATCH_BYTES < size(B + 1, n, k)
    g = torch.Generator(device="cuda")
    g.manual_seed(78)
    s = torch.randn(B + 1, n, generator=g, device="cuda")
    ref, got = _run_both(csa2, s[:B].contiguous(), k)
    assert torch.equal(ref, got)
    idx = torch.empty(B + 1, k, dtype=torch.int32, device="cuda")
    with pytest.raises(csa2.Csa2Error) as e:
        csa2.csa2_topk_static(s, k, idx)
    assert e.value.status == -8
    assert csa2.csa2_get_last_error() == 0
