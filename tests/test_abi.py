"""The C-ABI library builds, loads and exports every symbol include/dflash.h
declares.  Host-only: no CUDA compute call is made."""
import ctypes
import os

import pytest

from block_diffusion_speculative_hiddens_gb300 import _build, binding
from workload import CONFIGS


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_build.LIB):
        _build.build()
    return binding.load()


def test_every_declared_symbol_is_exported(lib):
    names = binding.declared_functions()
    assert len(names) >= 19
    assert set(names) == set(binding._SIGS), "binding and header disagree"
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code, text in binding.STATUS.items():
        assert lib.dflash_status_string(code).decode() == text
    assert lib.dflash_status_string(99).decode() == "unknown status"


def _cfg(c, **kw):
    d = dict(hidden=c.hidden, n_q_heads=c.n_q_heads, n_kv_heads=c.n_kv_heads, head_dim=c.head_dim,
             intermediate=c.intermediate, n_layers=c.n_layers, vocab=c.vocab, n_fused=c.n_fused,
             block=c.block, mask_id=c.mask_id, page_size=c.page_size, max_batch=c.batch,
             max_slots=c.batch, max_pages=64 * c.batch, max_pages_per_slot=64, max_rows=2048,
             device=0, rms_eps=c.rms_eps, rope_theta=c.rope_theta)
    d.update(kw)
    return binding.DflashConfig(**d)


@pytest.mark.parametrize("name", sorted(CONFIGS))
def test_workspace_sizing_accepts_every_workload(lib, name):
    n = lib.dflash_workspace_bytes(ctypes.byref(_cfg(CONFIGS[name])))
    assert n > 0 and n % 256 == 0


def test_target_role_accepted_with_enough_layers(lib):
    assert lib.dflash_workspace_bytes(ctypes.byref(_cfg(CONFIGS["tiny"], role=1, n_layers=8))) > 0
    assert lib.dflash_workspace_bytes(ctypes.byref(_cfg(CONFIGS["tiny"], role=1, n_layers=8, block=8))) == 0


@pytest.mark.parametrize("bad", [dict(head_dim=96), dict(block=1), dict(block=17), dict(page_size=32), dict(n_layers=9),
                                 dict(n_kv_heads=3), dict(max_batch=65), dict(mask_id=-1),
                                 dict(hidden=200), dict(rope_theta=0.5), dict(attn_impl=3), dict(role=2),
                                 dict(role=1)])
def test_workspace_sizing_rejects_unsupported(lib, bad):
    assert lib.dflash_workspace_bytes(ctypes.byref(_cfg(CONFIGS["tiny"], **bad))) == 0


def test_null_arguments_rejected_without_device(lib):
    # host-side checks return before any CUDA call
    assert lib.dflash_destroy(None) == 1
    assert lib.dflash_draft_block(None, None, 1, None, None, None) == 1
    assert lib.dflash_draft_block(None, None, 0, None, None, None) == 1
    assert lib.dflash_fuse_inject(None, None, 1, None, 16, None, None) == 1
    assert lib.dflash_draft_round(None, None, 1, None, 16, None, None, None, None) == 1
    assert lib.dflash_plan(None, None) == 1
    assert lib.dflash_verify_block(None, None, 1, None, None, None, None, None) == 1
    assert lib.dflash_advance(None, None, 1, None, None) == 1
    assert lib.dflash_accept_trim(None, None, 1, None, None, None, None, None, None) == 1
    assert lib.dflash_launch_count(None) == 0
    out = ctypes.c_void_p()
    assert lib.dflash_create(None, None, None, 0, ctypes.byref(out)) == 2
