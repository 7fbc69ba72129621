"""dflash_fuse_inject_noalloc against dflash_fuse_inject and the oracle.

The no-allocation variant serves callers that cannot hand the library any
extra device memory when they call it (their workspace was sized without
room for per-call scratch, or their device memory belongs to another
allocator); it keeps its scratch in a static array inside the library.  Two
slots of one handle receive the same features, one through each entry point,
over two calls in a row (a prefill chunk, then a round-sized append of fewer
rows than given); the injected K/V must agree with each other and with the
oracle's within the tolerance the parity tests use.  The shapes cover f16
and FP8 weights and the widest hidden sizes the static rows are sized for.
This file is collected last on purpose.
"""
import numpy as np
import pytest

from tests.gpu_util import TOL_REL_L2, rel_l2, to_np
from workload import feature_rows, get_config, make_weights

pytestmark = pytest.mark.gpu

CASES = [pytest.param("small", 0, id="small-f16"), pytest.param("small", 1, id="small-fp8"),
         pytest.param("wide-4096", 1, id="h4096-fp8"), pytest.param("wide-8192", 0, id="h8192-f16")]


@pytest.mark.parametrize("name,fp8", CASES)
def test_fuse_inject_noalloc_matches_fuse_inject_and_oracle(lib, name, fp8):
    import torch
    import oracle as O
    from block_diffusion_speculative_hiddens_gb300 import Drafter, weights_to_device
    from block_diffusion_speculative_hiddens_gb300.binding import DflashError

    cfg = get_config(name)
    w = make_weights(cfg)
    d = Drafter(cfg, weights_to_device(w), max_batch=4, max_slots=2, max_pages=8, max_pages_per_slot=4,
                max_rows=64, weight_fp8=fp8)
    dev = torch.device("cuda:0")
    i32 = dict(dtype=torch.int32, device=dev)
    F = cfg.fused_dim
    fr = feature_rows(cfg, 0, 0, 64)
    rows = torch.from_numpy(fr.reshape(64, F).view(np.int16)).view(torch.bfloat16).to(dev)

    # the oracle receives the same rows: 48, then the first 11 of the next 16
    orc = O.OracleDrafter(O.OracleModel(cfg, w, cache=True, fp8=bool(fp8)))
    req = O.OracleRequest(cfg, 64)
    calls = [(rows[None, :48], 48, 48, fr[:48]), (rows[None, 48:64], 16, 11, fr[48:59])]
    total = 0
    for feats, rpr, n, f_np in calls:
        n_new = torch.tensor([n], **i32)
        d.fuse_inject(torch.tensor([0], **i32), feats.contiguous(), rpr, n_new)
        d.fuse_inject_noalloc(torch.tensor([1], **i32), feats.contiguous(), rpr, n_new)
        orc.fuse_inject(req, f_np)
        total += n
        lens = to_np(d.slot_lengths(torch.tensor([0, 1], **i32)))
        assert lens.tolist() == [total, total]
        for l in range(cfg.n_layers):
            k0, v0 = d.read_kv(l, 0, 0, total)
            k1, v1 = d.read_kv(l, 1, 0, total)
            ok, ov = req.ctx(l)
            assert rel_l2(to_np(k1), to_np(k0)) < TOL_REL_L2, l
            assert rel_l2(to_np(v1), to_np(v0)) < TOL_REL_L2, l
            assert rel_l2(to_np(k1), ok) < TOL_REL_L2, l
            assert rel_l2(to_np(v1), ov) < TOL_REL_L2, l
    assert d.read_status() == 0

    # more rows than the static scratch holds: refused, nothing enqueued
    big = torch.zeros(1, 65, F, dtype=torch.bfloat16, device=dev)
    with pytest.raises(DflashError) as e:
        d.fuse_inject_noalloc(torch.tensor([1], **i32), big, 65, torch.tensor([65], **i32))
    assert e.value.code == 3
    assert to_np(d.slot_lengths(torch.tensor([1], **i32)))[0] == total
