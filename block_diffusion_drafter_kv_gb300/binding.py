"""ctypes binding of libdflash.so (include/dflash.h): argument marshalling only.

Every step of the draft-and-verify path runs in the library's CUDA kernels. PyTorch
supplies device memory and the current stream. If the shared library is missing the
import of `lib()` raises: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_float, c_int32, c_size_t, c_void_p
from typing import Optional

from .build import LIB_PATH

DFLASH_OK = 0
DFLASH_E_INVAL = -1
STATUS = {0: "ok", -1: "invalid argument", -2: "unsupported drafter shape", -3: "capacity exceeded",
          -4: "CUDA error", -5: "state not bound"}
DEV_TIMEOUT, DEV_CAPACITY, DEV_TOKEN = 1, 2, 4
OPT_WAIT_LIMIT_NS, OPT_CHAIN_MAX, OPT_GEMV_VARIANT, OPT_ATTN_SPLIT, OPT_ATTN_KEY_GROUPS = 1, 2, 3, 4, 5
OPT_INJECT_PASS_ROWS = 6
OPT_ATTN_MODE = 7


class DflashConfig(ctypes.Structure):
    _fields_ = [("hidden", c_int32), ("n_heads", c_int32), ("n_kv_heads", c_int32), ("head_dim", c_int32),
                ("n_layers", c_int32), ("intermediate", c_int32), ("vocab", c_int32), ("n_taps", c_int32),
                ("target_hidden", c_int32), ("rope_theta", c_float), ("rms_eps", c_float),
                ("max_block", c_int32), ("max_batch", c_int32), ("kv_capacity", c_int32)]


class DflashLayerWeights(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down", "g_attn", "g_mlp")]


class DflashWeights(ctypes.Structure):
    _fields_ = [("w_fc", c_void_p), ("g_ctx", c_void_p), ("embed", c_void_p), ("mask_emb", c_void_p),
                ("g_final", c_void_p), ("lm_head", c_void_p), ("layers", POINTER(DflashLayerWeights))]


# name -> (restype, argtypes); mirrors include/dflash.h
SIGNATURES = {
    "dflash_config_check": (c_int32, [POINTER(DflashConfig)]),
    "dflash_workspace_size": (c_size_t, [POINTER(DflashConfig)]),
    "dflash_create": (c_int32, [POINTER(DflashConfig), POINTER(DflashWeights), POINTER(c_void_p)]),
    "dflash_destroy": (c_int32, [c_void_p]),
    "dflash_bind_state": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t]),
    "dflash_bind_state_paged": (c_int32, [c_void_p, c_void_p, c_void_p, c_int32, c_void_p, c_int32, c_void_p,
                                          c_void_p, c_void_p, c_size_t]),
    "dflash_inject_ctx": (c_int32, [c_void_p, c_void_p, c_int32, c_void_p, c_int32, c_void_p]),
    "dflash_draft_block": (c_int32, [c_void_p, c_int32, c_int32, c_void_p, c_void_p, c_void_p, c_void_p]),
    "dflash_verify_greedy": (c_int32, [c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_void_p, c_void_p,
                                       c_void_p]),
    "dflash_verify_sampling": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, c_float, c_int32, c_int32, c_void_p,
                                         c_void_p, c_void_p]),
    "dflash_verify_greedy_hidden": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int32, c_int32,
                                              c_void_p, c_void_p, c_void_p]),
    "dflash_linear_bf16": (c_int32, [c_void_p, c_void_p, c_int32, c_int32, c_void_p, c_int32, c_void_p,
                                     c_void_p]),
    "dflash_read_device_error": (c_int32, [c_void_p, POINTER(c_int32), c_int32, c_void_p]),
    "dflash_set_option": (c_int32, [c_void_p, c_int32, ctypes.c_int64]),
    "dflash_get_option": (c_int32, [c_void_p, c_int32, POINTER(ctypes.c_int64)]),
    "dflash_selftest_timeout": (c_int32, [c_void_p, c_void_p]),
    "dflash_last_launch_count": (c_int32, [c_void_p]),
    "dflash_trace_events": (c_int32, [c_void_p, POINTER(c_void_p), c_int32]),
    "dflash_timeline": (c_int32, [c_void_p, c_void_p, ctypes.c_int64]),
    "dflash_timeline_used": (ctypes.c_int64, [c_void_p]),
    "dflash_status_string": (ctypes.c_char_p, [c_int32]),
    "dflash_verify_greedy_noalloc": (c_int32, [c_void_p, c_void_p, c_int32, c_int32, c_int32, c_void_p, c_void_p,
                                               c_void_p, c_void_p]),
    "dflash_synth_plant": (c_int32, [c_void_p, c_void_p, c_void_p, c_int32, c_void_p, c_int32, c_int32, c_int32,
                                     c_float, c_void_p, c_void_p]),
    "dflash_synth_unplant": (c_int32, [c_void_p, c_void_p, c_int32, c_int32, c_int32, c_void_p, c_void_p]),
}

_LIB = None


def lib(path: Optional[str] = None):
    """Load libdflash.so (built by `build.build()`); raises if it is absent."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libdflash.so not found at {p}: run block_diffusion_drafter_kv_gb300.build.build()")
    L = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    if path is None:
        _LIB = L
    return L


class DFlashError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS.get(status, status)} ({status})")
        self.status = status


def check(status: int, what: str) -> None:
    if status != DFLASH_OK:
        raise DFlashError(status, what)


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def make_config(shape, max_block: int, max_batch: int, kv_capacity: int) -> DflashConfig:
    return DflashConfig(shape.hidden, shape.n_heads, shape.n_kv_heads, shape.head_dim, shape.n_layers,
                        shape.intermediate, shape.vocab, shape.n_taps, shape.target_hidden,
                        float(shape.rope_theta), float(shape.rms_eps), max_block, max_batch, kv_capacity)


class Drafter:
    """One registered drafter plus its caller-owned state (KV caches, lengths, workspace).

    `weights` has the attributes of the input generator's `Weights` (bf16 CUDA tensors)."""

    def __init__(self, shape, weights, max_block: int, max_batch: int, kv_capacity: int, n_pages: int = 0,
                 page_table=None):
        """n_pages > 0 binds a paged KV cache: a pool of n_pages pages of 64 positions
        (k_cache / v_cache [L][n_pages * 64][nkv][d]) and `page_table`, an int32 CUDA tensor
        [max_batch][pages_per_seq] of page ids that the caller fills (and may change between
        calls)."""
        import torch
        self.L = lib()
        self.shape = shape
        self.cfg = make_config(shape, max_block, max_batch, kv_capacity)
        self.weights = weights  # keep the tensors alive
        lw = (DflashLayerWeights * shape.n_layers)()
        for i, w in enumerate(weights.layers):
            lw[i] = DflashLayerWeights(*[getattr(w, n).data_ptr() for n in
                                         ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down", "g_attn", "g_mlp")])
        self._lw = lw
        W = DflashWeights(weights.w_fc.data_ptr(), weights.g_ctx.data_ptr(), weights.embed.data_ptr(),
                          weights.mask_emb.data_ptr(), weights.g_final.data_ptr(), weights.lm_head.data_ptr(),
                          ctypes.cast(lw, POINTER(DflashLayerWeights)))
        h = c_void_p()
        check(self.L.dflash_create(ctypes.byref(self.cfg), ctypes.byref(W), ctypes.byref(h)), "dflash_create")
        self.h = h
        dev = weights.w_fc.device
        s = shape
        rows = (n_pages * 64,) if n_pages else (max_batch, kv_capacity)
        self.k_cache = torch.zeros(s.n_layers, *rows, s.n_kv_heads, s.head_dim, dtype=torch.float16, device=dev)
        self.v_cache = torch.zeros(s.n_layers, *rows, s.n_kv_heads, s.head_dim, dtype=torch.float16, device=dev)
        self.page_table = page_table
        self.len = torch.zeros(max_batch, dtype=torch.int32, device=dev)
        self.last_token = torch.zeros(max_batch, dtype=torch.int32, device=dev)
        nbytes = self.L.dflash_workspace_size(ctypes.byref(self.cfg))
        if nbytes == 0:
            raise DFlashError(-2, "dflash_workspace_size")
        self.workspace = torch.empty(nbytes + 256, dtype=torch.uint8, device=dev)
        base = self.workspace.data_ptr()
        self._ws_ptr = (base + 255) // 256 * 256
        if n_pages:
            assert page_table is not None and page_table.dtype == torch.int32 and page_table.is_cuda
            check(self.L.dflash_bind_state_paged(self.h, self.k_cache.data_ptr(), self.v_cache.data_ptr(), n_pages,
                                                 page_table.data_ptr(), page_table.shape[1], self.len.data_ptr(),
                                                 self.last_token.data_ptr(), self._ws_ptr, nbytes),
                  "dflash_bind_state_paged")
        else:
            check(self.L.dflash_bind_state(self.h, self.k_cache.data_ptr(), self.v_cache.data_ptr(),
                                           self.len.data_ptr(), self.last_token.data_ptr(), self._ws_ptr, nbytes),
                  "dflash_bind_state")

    # -- the three calls of the step ---------------------------------------------------
    def inject(self, hidden, rows_per_seq: int, n_new, batch: int, stream=None):
        import torch
        _require(hidden, torch.bfloat16, "hidden")
        _require(n_new, torch.int32, "n_new")
        check(self.L.dflash_inject_ctx(self.h, hidden.data_ptr(), rows_per_seq, n_new.data_ptr(), batch,
                                       _stream(stream)), "dflash_inject_ctx")

    def draft(self, batch: int, block: int, drafted, logits=None, x_trace=None, stream=None):
        import torch
        _require_opt(drafted, torch.int32, "drafted")
        _require_opt(logits, torch.float32, "logits")
        _require_opt(x_trace, torch.float32, "x_trace")
        check(self.L.dflash_draft_block(self.h, batch, block, _ptr(drafted), _ptr(logits), _ptr(x_trace),
                                        _stream(stream)), "dflash_draft_block")

    def verify(self, target_logits, drafted, batch: int, block: int, accept_len, committed, stream=None):
        import torch
        _require(target_logits, torch.float32, "target_logits")
        _require_opt(drafted, torch.int32, "drafted")
        _require(accept_len, torch.int32, "accept_len")
        _require(committed, torch.int32, "committed")
        check(self.L.dflash_verify_greedy(self.h, target_logits.data_ptr(), _ptr(drafted), batch, block,
                                          accept_len.data_ptr(), committed.data_ptr(), _stream(stream)),
              "dflash_verify_greedy")

    def verify_sampling(self, target_logits, drafted, uniforms, temperature: float, batch: int, block: int,
                        accept_len, committed, stream=None):
        """Speculative-sampling verification at `temperature` with caller-drawn uniforms
        (fp32 [batch][B]: accept tests, then the sampling draw)."""
        import torch
        _require(target_logits, torch.float32, "target_logits")
        _require_opt(drafted, torch.int32, "drafted")
        _require(uniforms, torch.float32, "uniforms")
        _require(accept_len, torch.int32, "accept_len")
        _require(committed, torch.int32, "committed")
        check(self.L.dflash_verify_sampling(self.h, target_logits.data_ptr(), _ptr(drafted), uniforms.data_ptr(),
                                            float(temperature), batch, block, accept_len.data_ptr(),
                                            committed.data_ptr(), _stream(stream)), "dflash_verify_sampling")

    def verify_hidden(self, target_hidden, target_gain, target_lm_head, drafted, batch: int, block: int, accept_len,
                      committed, stream=None):
        """Greedy verification from the target's last hidden states (bf16 [batch*B][Ht]), its
        final-norm gain (bf16 [Ht]) and LM head (bf16 [V][Ht])."""
        import torch
        for t, n in ((target_hidden, "target_hidden"), (target_gain, "target_gain"), (target_lm_head, "target_lm_head")):
            _require(t, torch.bfloat16, n)
        _require_opt(drafted, torch.int32, "drafted")
        _require(accept_len, torch.int32, "accept_len")
        _require(committed, torch.int32, "committed")
        check(self.L.dflash_verify_greedy_hidden(self.h, target_hidden.data_ptr(), target_gain.data_ptr(),
                                                 target_lm_head.data_ptr(), _ptr(drafted), batch, block,
                                                 accept_len.data_ptr(), committed.data_ptr(), _stream(stream)),
              "dflash_verify_greedy_hidden")

    # -- helpers -------------------------------------------------------------------------
    def linear(self, W, X, Y, stream=None):
        import torch
        _require(W, torch.bfloat16, "W")
        _require(X, torch.bfloat16, "X")
        _require(Y, torch.float32, "Y")
        check(self.L.dflash_linear_bf16(self.h, W.data_ptr(), W.shape[0], W.shape[1], X.data_ptr(), X.shape[0],
                                        Y.data_ptr(), _stream(stream)), "dflash_linear_bf16")

    def device_error(self, clear: bool = True, stream=None) -> int:
        """The device error flag once the work queued on `stream` (default: the current
        stream) has finished; with `clear`, the flag and the kernels' counters are reset."""
        f = c_int32(0)
        check(self.L.dflash_read_device_error(self.h, ctypes.byref(f), 1 if clear else 0, _stream(stream)),
              "dflash_read_device_error")
        return f.value

    def set_option(self, option: int, value: int) -> None:
        check(self.L.dflash_set_option(self.h, option, int(value)), "dflash_set_option")

    def get_option(self, option: int) -> int:
        v = ctypes.c_int64(0)
        check(self.L.dflash_get_option(self.h, option, ctypes.byref(v)), "dflash_get_option")
        return v.value

    def selftest_timeout(self, stream=None) -> None:
        check(self.L.dflash_selftest_timeout(self.h, _stream(stream)), "dflash_selftest_timeout")

    def last_launch_count(self) -> int:
        return self.L.dflash_last_launch_count(self.h)

    def timeline(self, records=None) -> None:
        """Per-CTA timeline into `records` (int64 CUDA tensor [n, 21]); None turns it off."""
        n = 0 if records is None else records.shape[0]
        self._tl_keep = records
        check(self.L.dflash_timeline(self.h, None if records is None else records.data_ptr(), n), "dflash_timeline")

    def timeline_used(self) -> int:
        return self.L.dflash_timeline_used(self.h)

    def trace_events(self, events) -> None:
        """Record torch.cuda.Event objects around each launch of later calls ([] turns it off)."""
        arr = (c_void_p * max(1, len(events)))(*[e.cuda_event for e in events])
        self._trace_keep = (arr, list(events))
        check(self.L.dflash_trace_events(self.h, arr, len(events)), "dflash_trace_events")

    def close(self):
        if getattr(self, "h", None):
            self.L.dflash_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _require(t, dtype, name):
    import torch
    if t.dtype != dtype or not t.is_cuda or not t.is_contiguous():
        raise DFlashError(DFLASH_E_INVAL, f"{name} must be a contiguous {dtype} CUDA tensor "
                                          f"(got {t.dtype}, cuda={t.is_cuda}, contiguous={t.is_contiguous()})")


def _require_opt(t, dtype, name):
    if t is not None:
        _require(t, dtype, name)


def verify_greedy_noalloc(target_logits, drafted, batch: int, block: int, accept_len, committed, last_token,
                          stream=None):
    """Greedy verification with no handle and no allocation (scratch is a fixed array in the library)."""
    import torch
    _require(target_logits, torch.float32, "target_logits")
    for t, n in ((accept_len, "accept_len"), (committed, "committed"), (last_token, "last_token")):
        _require(t, torch.int32, n)
    if drafted is not None:
        _require(drafted, torch.int32, "drafted")
    check(lib().dflash_verify_greedy_noalloc(target_logits.data_ptr(), _ptr(drafted), batch, block,
                                             target_logits.shape[-1], accept_len.data_ptr(), committed.data_ptr(),
                                             last_token.data_ptr(), _stream(stream)), "dflash_verify_greedy_noalloc")


def synth_plant(logits, drafted, masks, n_steps: int, step_counter, batch: int, block: int, bump: float, saved,
                stream=None):
    check(lib().dflash_synth_plant(logits.data_ptr(), _ptr(drafted), masks.data_ptr(), n_steps,
                                   step_counter.data_ptr(), batch, block, logits.shape[-1], bump, saved.data_ptr(),
                                   _stream(stream)), "dflash_synth_plant")


def synth_unplant(logits, step_counter, n_steps: int, batch: int, block: int, saved, stream=None):
    check(lib().dflash_synth_unplant(logits.data_ptr(), step_counter.data_ptr(), n_steps, batch, block,
                                     saved.data_ptr(), _stream(stream)), "dflash_synth_unplant")
