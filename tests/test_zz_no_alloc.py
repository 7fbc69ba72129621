"""dflash_fuse_inject_noalloc against dflash_fuse_inject.

The no-allocation variant serves callers that cannot hand the library any
extra device memory when they call it (their workspace was sized without
room for per-call scratch, or their device memory belongs to another
allocator); it keeps its scratch in a static array inside the library.  Two
slots of one handle receive the same features, one through each entry point,
over two calls in a row (a prefill chunk, then a round-sized append of fewer
rows than given); the injected K/V must agree within the tolerance the
parity tests use.  This file is collected last on purpose.
"""
import numpy as np
import pytest

from tests.gpu_util import TOL_REL_L2, rel_l2, to_np
from workload import feature_rows, get_config, make_weights

pytestmark = pytest.mark.gpu


def test_fuse_inject_noalloc_matches_fuse_inject(lib):
    import torch
    from block_diffusion_speculative_hiddens_gb300 import Drafter, weights_to_device
    from block_diffusion_speculative_hiddens_gb300.binding import DflashError

    cfg = get_config("small")
    d = Drafter(cfg, weights_to_device(make_weights(cfg)), max_batch=4, max_slots=2, max_pages=8,
                max_pages_per_slot=4, max_rows=64)
    dev = torch.device("cuda:0")
    i32 = dict(dtype=torch.int32, device=dev)
    F = cfg.fused_dim
    rows = torch.from_numpy(feature_rows(cfg, 0, 0, 64).reshape(64, F).view(np.int16)).view(torch.bfloat16).to(dev)

    calls = [(rows[None, :48], 48, 48), (rows[None, 48:64], 16, 11)]  # (features, rows_per_req, n_new)
    total = 0
    for feats, rpr, n in calls:
        n_new = torch.tensor([n], **i32)
        d.fuse_inject(torch.tensor([0], **i32), feats.contiguous(), rpr, n_new)
        d.fuse_inject_noalloc(torch.tensor([1], **i32), feats.contiguous(), rpr, n_new)
        total += n
        lens = to_np(d.slot_lengths(torch.tensor([0, 1], **i32)))
        assert lens.tolist() == [total, total]
        for l in range(cfg.n_layers):
            k0, v0 = d.read_kv(l, 0, 0, total)
            k1, v1 = d.read_kv(l, 1, 0, total)
            assert rel_l2(to_np(k1), to_np(k0)) < TOL_REL_L2, l
            assert rel_l2(to_np(v1), to_np(v0)) < TOL_REL_L2, l
    assert d.read_status() == 0

    # more rows than the static scratch holds: refused, nothing enqueued
    big = torch.zeros(1, 65, F, dtype=torch.bfloat16, device=dev)
    with pytest.raises(DflashError) as e:
        d.fuse_inject_noalloc(torch.tensor([1], **i32), big, 65, torch.tensor([65], **i32))
    assert e.value.code == 3
