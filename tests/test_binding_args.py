"""The Python binding refuses buffers a call would read or write past before
the library sees them (the C ABI only gets device pointers): wrong dtype,
device, layout or too few elements raise ValueError, and well-formed
arguments reach the library unchanged.  CPU only: tensors are stand-ins that
carry a CUDA device, and the library is a recorder."""
import types

import pytest
import torch

from block_diffusion_speculative_hiddens_gb300.binding import Drafter
from workload import get_config


class FakeT:
    def __init__(self, shape, dtype=torch.int32, device="cuda:0", contiguous=True):
        self.shape, self.dtype, self.device, self._c = tuple(shape), dtype, torch.device(device), contiguous

    def numel(self):
        n = 1
        for s in self.shape:
            n *= s
        return n

    def is_contiguous(self):
        return self._c

    def data_ptr(self):
        return 0x1000


class Recorder:
    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        def fn(*args):
            self.calls.append(name)
            return 0
        return fn


def _drafter(name="tiny"):
    d = Drafter.__new__(Drafter)
    d.cfg, d.device, d.lib, d.h = get_config(name), 0, Recorder(), None
    return d


STREAM = types.SimpleNamespace(cuda_stream=0)
B = 2


def test_well_formed_round_reaches_the_library():
    d = _drafter()
    cfg = d.cfg
    F, S = cfg.n_fused * cfg.hidden, cfg.block
    slots = FakeT([B])
    d.fuse_inject(slots, FakeT([B, S, F], torch.bfloat16), S, FakeT([B]), STREAM)
    d.draft_block(slots, FakeT([B]), FakeT([B, S - 1]), STREAM)
    d.draft_block_debug(slots, FakeT([B]), FakeT([B, S - 1]), FakeT([B * 16, cfg.hidden], torch.float32),
                        FakeT([B * 16, cfg.vocab], torch.float32), STREAM)
    d.draft_block_sample(slots, FakeT([B]), 1.0, 3, FakeT([1]), FakeT([B, S - 1]), None, STREAM)
    d.accept_trim(slots, FakeT([B, S - 1]), FakeT([B, S]), FakeT([B]), FakeT([B]), FakeT([B]), STREAM)
    d.verify_block(slots, FakeT([B, 16]), FakeT([B, 16]), None, FakeT([B, 16, F], torch.bfloat16), STREAM)
    d.advance(slots, FakeT([B]), STREAM)
    d.fuse_inject(FakeT([0]), None, 0, FakeT([0]), STREAM)  # an empty batch touches nothing
    assert d.lib.calls == ["dflash_fuse_inject", "dflash_draft_block", "dflash_draft_block_debug",
                           "dflash_draft_block_sample", "dflash_accept_trim", "dflash_verify_block",
                           "dflash_advance", "dflash_fuse_inject"]


@pytest.mark.parametrize("bad", ["short", "dtype", "device", "host", "strided", "missing"])
def test_bad_buffers_are_refused_before_the_library(bad):
    d = _drafter()
    S = d.cfg.block
    kw = dict(shape=[B, S - 1])
    if bad == "short":
        kw["shape"] = [B, S - 2]
    draft = FakeT(**kw)
    if bad == "dtype":
        draft = FakeT([B, S - 1], torch.int64)
    elif bad == "device":
        draft = FakeT([B, S - 1], device="cuda:1")
    elif bad == "host":
        draft = FakeT([B, S - 1], device="cpu")
    elif bad == "strided":
        draft = FakeT([B, S - 1], contiguous=False)
    elif bad == "missing":
        draft = None
    with pytest.raises(ValueError):
        d.draft_block(FakeT([B]), FakeT([B]), draft, STREAM)
    assert d.lib.calls == []


def test_feature_rows_sized_by_rows_per_request():
    d = _drafter()
    F = d.cfg.n_fused * d.cfg.hidden
    with pytest.raises(ValueError):
        d.fuse_inject(FakeT([B]), FakeT([B, 7, F], torch.bfloat16), 8, FakeT([B]), STREAM)
    with pytest.raises(ValueError):  # rows to read but no buffer
        d.fuse_inject(FakeT([B]), None, 8, FakeT([B]), STREAM)
    with pytest.raises(ValueError):  # the debug outputs hold all 16 rows of a request
        d.draft_block_debug(FakeT([B]), FakeT([B]), FakeT([B, d.cfg.block - 1]),
                            FakeT([B * d.cfg.block - 1, d.cfg.hidden], torch.float32), None, STREAM)
    assert d.lib.calls == []
