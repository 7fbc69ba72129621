"""ctypes binding of libdflash (include/dflash.h): argument marshalling only.

Every compute step runs in the CUDA library; this module turns torch tensors
into device pointers and CUDA streams into handles.  Loading fails loudly if
the library is missing or was built without the expected symbols -- there is
no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libdflash.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "dflash.h")

OK = 0
STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported shape", 3: "capacity exceeded",
          4: "CUDA error", 5: "device-side check failed", 6: "workspace too small or misaligned",
          7: "a weight exceeds the f16 range"}
DEV_TIMEOUT, DEV_NAN, DEV_PAGE, DEV_CAPACITY, DEV_ARG, DEV_RANGE = 0x01, 0x02, 0x04, 0x08, 0x10, 0x20
KID_LM_HEAD, KID_GATE_UP, KID_ATTENTION, KID_DOWN, KID_QKV, KID_WO, KID_FC, KID_INJECT = 1, 2, 3, 4, 5, 6, 7, 8
KID_ALL = 255  # trace_arm: every GEMM and attention launch in turn

_c_int_p = ctypes.POINTER(ctypes.c_int32)
_vp = ctypes.c_void_p


class DflashConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "hidden", "n_q_heads", "n_kv_heads", "head_dim", "intermediate", "n_layers", "vocab",
        "n_fused", "block", "mask_id", "page_size", "max_batch", "max_slots", "max_pages",
        "max_pages_per_slot", "max_rows", "device")] + [("rms_eps", ctypes.c_float),
                                                         ("rope_theta", ctypes.c_float),
                                                         ("attn_impl", ctypes.c_int32),
                                                         ("role", ctypes.c_int32),
                                                         ("weight_fp8", ctypes.c_int32)]


class DflashWeights(ctypes.Structure):
    _fields_ = [("embed", _vp), ("fc", _vp), ("fc_norm", _vp), ("final_norm", _vp)] + [
        (n, ctypes.POINTER(_vp)) for n in (
            "in_norm", "wqkv", "q_norm", "k_norm", "wo", "post_norm", "w_gate_up", "w_down")]


def declared_functions(header: str = HEADER):
    """Names of the functions include/dflash.h declares."""
    with open(header) as f:
        text = f.read()
    return sorted(set(re.findall(r"DFLASH_API\s+[\w\s\*]+?\b(dflash_\w+)\s*\(", text)))


_SIGS = {
    "dflash_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(DflashConfig)]),
    "dflash_create": (ctypes.c_int, [ctypes.POINTER(DflashConfig), ctypes.POINTER(DflashWeights), _vp,
                                     ctypes.c_size_t, ctypes.POINTER(_vp)]),
    "dflash_destroy": (ctypes.c_int, [_vp]),
    "dflash_fuse_inject": (ctypes.c_int, [_vp, _vp, ctypes.c_int32, _vp, ctypes.c_int32, _vp, _vp]),
    "dflash_fuse_inject_noalloc": (ctypes.c_int, [_vp, _vp, ctypes.c_int32, _vp, ctypes.c_int32, _vp, _vp]),
    "dflash_draft_block": (ctypes.c_int, [_vp, _vp, ctypes.c_int32, _vp, _vp, _vp]),
    "dflash_draft_round": (ctypes.c_int, [_vp, _vp, ctypes.c_int32, _vp, ctypes.c_int32, _vp, _vp, _vp, _vp]),
    "dflash_draft_block_debug": (ctypes.c_int, [_vp, _vp, ctypes.c_int32, _vp, _vp, _vp, _vp, _vp]),
    "dflash_draft_block_sample": (ctypes.c_int, [_vp, _vp, ctypes.c_int32, _vp, ctypes.c_float, ctypes.c_uint64,
                                                 _vp, _vp, _vp, _vp]),
    "dflash_accept_trim": (ctypes.c_int, [_vp, _vp, ctypes.c_int32, _vp, _vp, _vp, _vp, _vp, _vp]),
    "dflash_reset_slot": (ctypes.c_int, [_vp, ctypes.c_int32, _vp]),
    "dflash_check_wait_timeout": (ctypes.c_int, [_vp, ctypes.c_uint32, _vp]),
    "dflash_read_status": (ctypes.c_int, [_vp, ctypes.POINTER(ctypes.c_uint32)]),
    "dflash_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "dflash_graph_begin": (ctypes.c_int, [_vp, _vp]),
    "dflash_graph_end": (ctypes.c_int, [_vp, _vp, _c_int_p]),
    "dflash_graph_launch": (ctypes.c_int, [_vp, _vp]),
    "dflash_read_kv": (ctypes.c_int, [_vp, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                      _vp, _vp, _vp]),
    "dflash_slot_lengths": (ctypes.c_int, [_vp, _vp, ctypes.c_int32, _vp, _vp]),
    "dflash_probe_arm": (ctypes.c_int, [_vp, ctypes.c_int32, ctypes.c_int32]),
    "dflash_probe_read": (ctypes.c_int, [_vp, ctypes.POINTER(ctypes.c_float), ctypes.c_int32, _c_int_p]),
    "dflash_marks_arm": (ctypes.c_int, [_vp, ctypes.c_int32]),
    "dflash_mark": (ctypes.c_int, [_vp, _vp]),
    "dflash_marks_read": (ctypes.c_int, [_vp, _vp, ctypes.c_int32, _vp]),
    "dflash_launch_count": (ctypes.c_uint64, [_vp]),
    "dflash_plan": (ctypes.c_int, [_vp, _vp]),
    "dflash_verify_block": (ctypes.c_int, [_vp, _vp, ctypes.c_int32, _vp, _vp, _vp, _vp, _vp]),
    "dflash_advance": (ctypes.c_int, [_vp, _vp, ctypes.c_int32, _vp, _vp]),
    "dflash_verify_block_sample": (ctypes.c_int, [_vp, _vp, ctypes.c_int32, _vp, _vp, ctypes.c_float,
                                                  ctypes.c_uint64, _vp, _vp, _vp]),
    "dflash_trace_arm": (ctypes.c_int, [_vp, ctypes.c_int32, _vp, ctypes.c_int32]),
    "dflash_stamps_arm": (ctypes.c_int, [_vp, _vp, ctypes.c_int32]),
    "dflash_harness_verify": (ctypes.c_int, [_vp, _vp, ctypes.c_int32, _vp, _vp, _vp, ctypes.c_int32, _vp,
                                             _vp, _vp, ctypes.c_int32, _vp, _vp]),
}

_LIB = None


def load(path: str = LIB_PATH):
    """Load libdflash and declare every entry point's signature."""
    global _LIB
    if _LIB is not None and path == LIB_PATH:
        return _LIB
    if not os.path.exists(path):
        raise RuntimeError(f"libdflash not built ({path} missing): run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)  # AttributeError if the symbol is missing
        fn.restype = res
        fn.argtypes = args
    if path == LIB_PATH:
        _LIB = lib
    return lib


class DflashError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {STATUS.get(code, code)} ({code})")
        self.code = code


def _check(fn: str, code: int):
    if code != OK:
        raise DflashError(fn, code)


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _need(t, dtype: str, n: int, what: str, device: int, optional: bool = False):
    """Refuse a buffer the call would read or write past, before the library
    sees it: the C ABI gets a bare device pointer.  `n` elements of `dtype`
    (a torch dtype name), contiguous, on CUDA device `device`; nothing is
    checked when the call touches no element (n == 0) or an optional buffer
    is absent."""
    if n <= 0 or (t is None and optional):
        return
    if t is None:
        raise ValueError(f"{what}: a device tensor is required")
    dev = t.device
    if dev.type != "cuda" or dev.index != device:
        raise ValueError(f"{what}: expected a tensor on cuda:{device}, got {dev}")
    if str(t.dtype) != "torch." + dtype:
        raise ValueError(f"{what}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{what}: expected a contiguous tensor")
    if t.numel() < n:
        raise ValueError(f"{what}: {t.numel()} elements, the call needs {n}")


def _stream(stream) -> int:
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


class Drafter:
    """One libdflash handle: drafter weights (device), workspace and slots.

    `weights` follows workload.make_weights' layout with torch bf16 device
    tensors.  dflash_create copies them into the handle's workspace, so the
    caller may drop them afterwards.
    """

    def __init__(self, cfg, weights: dict, *, max_batch: int, max_slots: int, max_pages: int,
                 max_pages_per_slot: int, max_rows: int, device: int = 0, attn_impl: int = 0, role: int = 0,
                 weight_fp8: int = 0):
        import torch
        self.lib = load()
        self.cfg = cfg
        self.device = device
        self.w = weights
        self.role = role
        L = len(weights["layers"]) if role == 1 else cfg.n_layers
        self.n_layers = L
        c = DflashConfig(hidden=cfg.hidden, n_q_heads=cfg.n_q_heads, n_kv_heads=cfg.n_kv_heads,
                         head_dim=cfg.head_dim, intermediate=cfg.intermediate, n_layers=L,
                         vocab=cfg.vocab, n_fused=cfg.n_fused, block=cfg.block, mask_id=cfg.mask_id,
                         page_size=cfg.page_size, max_batch=max_batch, max_slots=max_slots,
                         max_pages=max_pages, max_pages_per_slot=max_pages_per_slot,
                         max_rows=max_rows, device=device, rms_eps=cfg.rms_eps,
                         rope_theta=cfg.rope_theta, attn_impl=attn_impl, role=role, weight_fp8=weight_fp8)
        self.c = c
        nbytes = self.lib.dflash_workspace_bytes(ctypes.byref(c))
        if nbytes == 0:
            raise DflashError("dflash_workspace_bytes", 2)
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=f"cuda:{device}")

        def arr(name):
            a = (_vp * L)(*[weights["layers"][l][name].data_ptr() for l in range(L)])
            return a

        self._arrays = {n: arr(n) for n in ("in_norm", "wqkv", "q_norm", "k_norm", "wo", "post_norm",
                                            "w_gate_up", "w_down")}
        opt = lambda n: weights[n].data_ptr() if n in weights else None  # noqa: E731  (no fusion in a target)
        wts = DflashWeights(embed=weights["embed"].data_ptr(), fc=opt("fc"), fc_norm=opt("fc_norm"),
                            final_norm=weights["final_norm"].data_ptr(),
                            **{n: ctypes.cast(a, ctypes.POINTER(_vp)) for n, a in self._arrays.items()})
        h = _vp()
        _check("dflash_create", self.lib.dflash_create(ctypes.byref(c), ctypes.byref(wts),
                                                       self.workspace.data_ptr(), nbytes,
                                                       ctypes.byref(h)))
        self.h = h
        self.max_batch, self.max_rows = max_batch, max_rows

    def close(self):
        if getattr(self, "h", None):
            self.lib.dflash_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ---- argument checks (sizes from include/dflash.h)
    def _inject_args(self, slots, feats, rows_per_req: int, n_new) -> int:
        B = slots.numel()
        _need(slots, "int32", B, "slots", self.device)
        _need(feats, "bfloat16", B * rows_per_req * self.cfg.n_fused * self.cfg.hidden, "feats", self.device)
        _need(n_new, "int32", B, "n_new", self.device)
        if B * rows_per_req > 0 and feats.data_ptr() % 16:
            raise ValueError("feats: the rows are read by a TMA descriptor and must start 16-byte aligned")
        return B

    def _draft_args(self, slots, last_tok, draft) -> int:
        B = slots.numel()
        _need(slots, "int32", B, "slots", self.device)
        _need(last_tok, "int32", B, "last_tok", self.device)
        _need(draft, "int32", B * (self.cfg.block - 1), "draft", self.device)
        return B

    # ---- the three calls of a round
    def fuse_inject(self, slots, feats, rows_per_req: int, n_new, stream=None):
        self._inject_args(slots, feats, rows_per_req, n_new)
        _check("dflash_fuse_inject", self.lib.dflash_fuse_inject(
            self.h, _ptr(slots), slots.numel(), _ptr(feats), rows_per_req, _ptr(n_new), _stream(stream)))

    def fuse_inject_noalloc(self, slots, feats, rows_per_req: int, n_new, stream=None):
        """dflash_fuse_inject with the library's static scratch (at most 64 rows)."""
        self._inject_args(slots, feats, rows_per_req, n_new)
        _check("dflash_fuse_inject_noalloc", self.lib.dflash_fuse_inject_noalloc(
            self.h, _ptr(slots), slots.numel(), _ptr(feats), rows_per_req, _ptr(n_new), _stream(stream)))

    def draft_block(self, slots, last_tok, draft, stream=None):
        self._draft_args(slots, last_tok, draft)
        _check("dflash_draft_block", self.lib.dflash_draft_block(
            self.h, _ptr(slots), slots.numel(), _ptr(last_tok), _ptr(draft), _stream(stream)))

    def draft_round(self, slots, feats, rows_per_req: int, n_new, last_tok, draft, stream=None):
        """fuse_inject + draft_block with the injection folded into the layers' QKV GEMMs."""
        self._inject_args(slots, feats, rows_per_req, n_new)
        self._draft_args(slots, last_tok, draft)
        _check("dflash_draft_round", self.lib.dflash_draft_round(
            self.h, _ptr(slots), slots.numel(), _ptr(feats), rows_per_req, _ptr(n_new), _ptr(last_tok),
            _ptr(draft), _stream(stream)))

    def draft_block_debug(self, slots, last_tok, draft, hidden=None, logits=None, stream=None):
        """hidden [batch*16, H] and logits [batch*16, V] float32: all 16 rows of each request."""
        B = self._draft_args(slots, last_tok, draft)
        _need(hidden, "float32", B * 16 * self.cfg.hidden, "hidden", self.device, optional=True)
        _need(logits, "float32", B * 16 * self.cfg.vocab, "logits", self.device, optional=True)
        _check("dflash_draft_block_debug", self.lib.dflash_draft_block_debug(
            self.h, _ptr(slots), slots.numel(), _ptr(last_tok), _ptr(draft), _ptr(hidden),
            _ptr(logits), _stream(stream)))

    def draft_block_sample(self, slots, last_tok, temperature: float, seed: int, round_ctr, draft, logits=None,
                           stream=None):
        """dflash_draft_block with each draft drawn from softmax(logits / temperature)."""
        B = self._draft_args(slots, last_tok, draft)
        _need(round_ctr, "int32", 1, "round_ctr", self.device, optional=True)
        _need(logits, "float32", B * 16 * self.cfg.vocab, "logits", self.device, optional=True)
        _check("dflash_draft_block_sample", self.lib.dflash_draft_block_sample(
            self.h, _ptr(slots), slots.numel(), _ptr(last_tok), float(temperature), int(seed) & ((1 << 64) - 1),
            _ptr(round_ctr), _ptr(draft), _ptr(logits), _stream(stream)))

    # ---- target model (role 1)
    def verify_block(self, slots, tokens, out_tok, n_valid=None, feats=None, stream=None):
        """Target forward over block tokens [batch, 16] -> out_tok [batch, 16] (+ feats [batch, 16, 5H])."""
        B = slots.numel()
        _need(slots, "int32", B, "slots", self.device)
        _need(tokens, "int32", B * 16, "tokens", self.device)
        _need(out_tok, "int32", B * 16, "out_tok", self.device)
        _need(n_valid, "int32", B, "n_valid", self.device, optional=True)
        _need(feats, "bfloat16", B * 16 * self.cfg.n_fused * self.cfg.hidden, "feats", self.device, optional=True)
        _check("dflash_verify_block", self.lib.dflash_verify_block(
            self.h, _ptr(slots), slots.numel(), _ptr(tokens), _ptr(n_valid), _ptr(out_tok), _ptr(feats),
            _stream(stream)))

    def verify_block_sample(self, slots, tokens, out_tok, temperature: float, seed: int, n_valid=None, feats=None,
                            stream=None):
        """verify_block with every row's token drawn from softmax(logits / temperature),
        keyed by (seed, slot, position)."""
        B = slots.numel()
        _need(slots, "int32", B, "slots", self.device)
        _need(tokens, "int32", B * 16, "tokens", self.device)
        _need(out_tok, "int32", B * 16, "out_tok", self.device)
        _need(n_valid, "int32", B, "n_valid", self.device, optional=True)
        _need(feats, "bfloat16", B * 16 * self.cfg.n_fused * self.cfg.hidden, "feats", self.device, optional=True)
        _check("dflash_verify_block_sample", self.lib.dflash_verify_block_sample(
            self.h, _ptr(slots), slots.numel(), _ptr(tokens), _ptr(n_valid), float(temperature),
            int(seed) & ((1 << 64) - 1), _ptr(out_tok), _ptr(feats), _stream(stream)))

    def advance(self, slots, n, stream=None):
        """ctx_len[slot] += n[b] (the trim after acceptance / a prefill chunk's step)."""
        B = slots.numel()
        _need(slots, "int32", B, "slots", self.device)
        _need(n, "int32", B, "n", self.device)
        _check("dflash_advance", self.lib.dflash_advance(self.h, _ptr(slots), slots.numel(), _ptr(n),
                                                          _stream(stream)))

    def accept_trim(self, slots, draft, target, accept_len, bonus, ctx_len, stream=None):
        B, S = slots.numel(), self.cfg.block
        _need(slots, "int32", B, "slots", self.device)
        _need(draft, "int32", B * (S - 1), "draft", self.device)
        _need(target, "int32", B * S, "target", self.device)
        for name, t in (("accept_len", accept_len), ("bonus", bonus), ("ctx_len", ctx_len)):
            _need(t, "int32", B, name, self.device)
        _check("dflash_accept_trim", self.lib.dflash_accept_trim(
            self.h, _ptr(slots), slots.numel(), _ptr(draft), _ptr(target), _ptr(accept_len),
            _ptr(bonus), _ptr(ctx_len), _stream(stream)))

    def check_wait_timeout(self, limit_us: int, stream=None):
        """Make one bounded in-kernel wait run out (nothing arrives at its barrier)."""
        _check("dflash_check_wait_timeout", self.lib.dflash_check_wait_timeout(self.h, int(limit_us),
                                                                               _stream(stream)))

    def reset_slot(self, slot: int, stream=None):
        _check("dflash_reset_slot", self.lib.dflash_reset_slot(self.h, slot, _stream(stream)))

    def read_status(self) -> int:
        v = ctypes.c_uint32(0)
        _check("dflash_read_status", self.lib.dflash_read_status(self.h, ctypes.byref(v)))
        return v.value

    # ---- introspection
    def read_kv(self, layer: int, slot: int, pos0: int, n: int, stream=None):
        import torch
        shape = (n, self.cfg.n_kv_heads, self.cfg.head_dim)
        k = torch.empty(shape, dtype=torch.float32, device=f"cuda:{self.device}")
        v = torch.empty_like(k)
        _check("dflash_read_kv", self.lib.dflash_read_kv(self.h, layer, slot, pos0, n, _ptr(k), _ptr(v),
                                                         _stream(stream)))
        return k, v

    def slot_lengths(self, slots, stream=None):
        import torch
        out = torch.empty(slots.numel(), dtype=torch.int32, device=slots.device)
        _check("dflash_slot_lengths", self.lib.dflash_slot_lengths(self.h, _ptr(slots), slots.numel(),
                                                                   _ptr(out), _stream(stream)))
        return out

    # ---- runtime
    def graph_begin(self, stream=None):
        _check("dflash_graph_begin", self.lib.dflash_graph_begin(self.h, _stream(stream)))

    def graph_end(self, stream=None) -> int:
        n = ctypes.c_int32(0)
        _check("dflash_graph_end", self.lib.dflash_graph_end(self.h, _stream(stream), ctypes.byref(n)))
        return n.value

    def graph_launch(self, stream=None):
        _check("dflash_graph_launch", self.lib.dflash_graph_launch(self.h, _stream(stream)))

    def probe_arm(self, kernel_id: int, n: int):
        _check("dflash_probe_arm", self.lib.dflash_probe_arm(self.h, kernel_id, n))

    def probe_read(self, cap: int):
        buf = (ctypes.c_float * max(cap, 1))()
        n = ctypes.c_int32(0)
        _check("dflash_probe_read", self.lib.dflash_probe_read(self.h, buf, cap, ctypes.byref(n)))
        return list(buf[:n.value])

    def marks_arm(self, n: int):
        _check("dflash_marks_arm", self.lib.dflash_marks_arm(self.h, n))

    def mark(self, stream=None):
        """Record the next timeline mark on the stream (a graph node when capturing)."""
        _check("dflash_mark", self.lib.dflash_mark(self.h, _stream(stream)))

    def marks_read(self, cap: int):
        """Intervals in ms between consecutive recorded marks (synchronises)."""
        buf = (ctypes.c_float * max(cap, 1))()
        n = ctypes.c_int32(0)
        _check("dflash_marks_read", self.lib.dflash_marks_read(self.h, buf, cap, ctypes.byref(n)))
        return list(buf[:n.value])

    def trace_arm(self, kernel_id: int, buf=None, cap_ctas: int = 0):
        """Arm a per-CTA timeline of the next launch of a GEMM kernel; buf is an
        int64 device tensor [cap_ctas, 8]."""
        _check("dflash_trace_arm", self.lib.dflash_trace_arm(self.h, kernel_id, _ptr(buf), cap_ctas))

    def stamps_arm(self, buf=None, n: int = 0):
        """Device timestamps of the next n stand-in verify calls into buf
        (int64 device tensor [n, 2]: start, end in ns)."""
        if n > 0:
            _need(buf, "int64", 2 * n, "stamps", self.device)
        _check("dflash_stamps_arm", self.lib.dflash_stamps_arm(self.h, _ptr(buf) if n > 0 else None, n))

    def launch_count(self) -> int:
        return int(self.lib.dflash_launch_count(self.h))

    def plan(self) -> dict:
        """SMs, attention splits and page loop, GEMM cluster size chosen at create."""
        v = (ctypes.c_int32 * 5)()
        _check("dflash_plan", self.lib.dflash_plan(self.h, v))
        return {"sms": v[0], "attn_splits": v[1], "attn_impl": ["", "warp MMAs", "tcgen05"][v[2]],
                "gemm_cluster": v[3], "attn_merge": ["cluster", "global"][v[4]]}

    def harness_verify(self, slots, draft, match, offs, rounds_cap: int, round_ctr, target,
                       feat_stream=None, stream_rows: int = 0, feats_out=None, stream=None):
        _check("dflash_harness_verify", self.lib.dflash_harness_verify(
            self.h, _ptr(slots), slots.numel(), _ptr(draft), _ptr(match), _ptr(offs), rounds_cap,
            _ptr(round_ctr), _ptr(target), _ptr(feat_stream), stream_rows, _ptr(feats_out),
            _stream(stream)))


def weights_to_device(w_np: dict, device: int = 0) -> dict:
    """workload.make_weights output (uint16 bf16 bits) -> torch bf16 tensors on the GPU."""
    import numpy as np
    import torch

    def t(a):
        a = np.ascontiguousarray(a)
        if not a.flags.writeable:  # memory-mapped cache files: copy once instead of aliasing read-only memory
            a = a.copy()
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(f"cuda:{device}")

    out = {k: t(v) for k, v in w_np.items() if k != "layers"}
    out["layers"] = [{k: t(v) for k, v in lw.items()} for lw in w_np["layers"]]
    return out


def bf16_host(a) -> "torch.Tensor":
    """uint16 bf16 bit patterns (numpy) -> torch bf16 CPU tensor (no copy of values)."""
    import numpy as np
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
