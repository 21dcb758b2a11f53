"""ctypes binding of libsmp (include/smp.h).  Argument marshalling only."""
import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
lib_path = os.path.join(HERE, "libsmp.so")

SMP_OK, SMP_ERR_EMPTY, SMP_ERR_NONFINITE, SMP_ERR_INVALID_PARAM = 0, 1, 2, 3
SMP_ERR_TIMEOUT, SMP_ERR_CUDA, SMP_ERR_CAPACITY = 4, 5, 6
SMP_F32, SMP_BF16, SMP_F16 = 0, 1, 2
SMP_KERNEL_BOARD, SMP_KERNEL_SPLIT = 0, 1
PATH_NAMES = {0: "error", 1: "greedy", 2: "all", 3: "sigma", 4: "full"}

_DTYPES = {torch.float32: SMP_F32, torch.bfloat16: SMP_BF16, torch.float16: SMP_F16}

EXPORTS = ("smp_create", "smp_destroy", "smp_topk_topp_mask", "smp_sample", "smp_argmax",
           "smp_sample_noalloc", "smp_sample_logprob", "smp_spec_verify",
           "smp_repetition_penalty", "smp_gumbel_sample", "smp_top_logprobs", "smp_set_row_info",
           "smp_set_kernel", "smp_set_wait_limit", "smp_plan",
           "smp_status_string")


class SmpError(RuntimeError):
    def __init__(self, code, what):
        super().__init__(f"{what}: status {code}")
        self.code = code


class RowParams(ctypes.Structure):
    _fields_ = [("temperature", ctypes.c_void_p), ("top_k", ctypes.c_void_p),
                ("top_p", ctypes.c_void_p), ("seed", ctypes.c_void_p),
                ("offset", ctypes.c_void_p)]


_lib = None


def load_library(path=None):
    """Load libsmp.so; raises if it has not been built."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or lib_path
    if not os.path.exists(p):
        raise FileNotFoundError(
            f"{p} is missing: build it with __graft_entry__.build() (nvcc, sm_103a)")
    L = ctypes.CDLL(p)
    P, I = ctypes.c_void_p, ctypes.c_int
    L.smp_create.argtypes = [ctypes.POINTER(P), I, I, I]
    L.smp_destroy.argtypes = [P]
    L.smp_topk_topp_mask.argtypes = [P, P, I, I, I, ctypes.c_int64, P, ctypes.POINTER(RowParams),
                                     P, P, P, P, P]
    L.smp_sample.argtypes = [P, P, I, I, I, ctypes.c_int64, P, ctypes.POINTER(RowParams), P, P,
                             P, P, P]
    L.smp_argmax.argtypes = [P, P, I, I, I, ctypes.c_int64, P, P, P, P]
    L.smp_sample_logprob.argtypes = [P, P, I, I, I, ctypes.c_int64, P,
                                     ctypes.POINTER(RowParams), P, P, P, P, P, P]
    L.smp_sample_noalloc.argtypes = [P, I, I, I, ctypes.c_int64, P, ctypes.POINTER(RowParams), P,
                                     P, P, P, P]
    L.smp_spec_verify.argtypes = [P, P, P, P, I, I, I, ctypes.c_int64, P, P, P, P, P, P]
    L.smp_repetition_penalty.argtypes = [P, P, I, I, I, ctypes.c_int64, P, I, ctypes.c_int64, P,
                                         P, P]
    L.smp_gumbel_sample.argtypes = [P, P, I, I, I, ctypes.c_int64, P, P, P, P, P, P, P]
    L.smp_top_logprobs.argtypes = [P, P, I, I, I, ctypes.c_int64, P, P, P, P, I, P, P, P]
    L.smp_set_row_info.argtypes = [P, P]
    L.smp_set_kernel.argtypes = [P, ctypes.c_int]
    L.smp_set_wait_limit.argtypes = [P, ctypes.c_longlong]
    L.smp_plan.argtypes = [P, I, I, I, ctypes.POINTER(I), ctypes.POINTER(I), ctypes.POINTER(I),
                           ctypes.POINTER(I)]
    L.smp_status_string.restype = ctypes.c_char_p
    L.smp_status_string.argtypes = [I]
    for name in EXPORTS:
        getattr(L, name).restype = getattr(L, name).restype or ctypes.c_int
    if path is None:
        _lib = L
    return L


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(rc, what):
    if rc != SMP_OK:
        raise SmpError(rc, what)


class Sampler:
    """A libsmp handle bound to one CUDA device.

    All tensors must be contiguous CUDA tensors on that device.  logits:
    [B, V] (or [B, ld] with ld >= V via ``ld``) float32 / bfloat16 / float16;
    bitmask: int32 [B, ceil(V/32)] holding uint32 bit patterns, or None;
    temperature float32 [B]; top_k int32 [B]; top_p float32 [B]; seed, offset
    int64 [B] holding uint64 bit patterns.
    """

    def __init__(self, device=0, max_batch=4096, max_vocab=1 << 20, lib=None):
        self.lib = lib or load_library()
        self.device = torch.device("cuda", device) if isinstance(device, int) else device
        h = ctypes.c_void_p()
        _check(self.lib.smp_create(ctypes.byref(h), self.device.index or 0, max_batch, max_vocab),
               "smp_create")
        self.h = h
        self._row_info = None

    def close(self):
        if getattr(self, "h", None):
            self.lib.smp_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- helpers ----------------------------------------------------------------
    def _stream(self):
        return ctypes.c_void_p(torch.cuda.current_stream(self.device).cuda_stream)

    def _check_tensor(self, t, name, dtype=None):
        if t is None:
            return
        if not t.is_cuda or t.device != self.device:
            raise ValueError(f"{name} must be on {self.device}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if dtype is not None and t.dtype != dtype:
            raise ValueError(f"{name} must be {dtype}, got {t.dtype}")

    def _prep(self, logits, V, bitmask, temperature, top_k, top_p, seed, offset):
        if logits.dtype not in _DTYPES:
            raise ValueError(f"unsupported logits dtype {logits.dtype}")
        self._check_tensor(logits, "logits")
        B, ld = logits.shape
        V = ld if V is None else V
        self._check_tensor(bitmask, "bitmask", torch.int32)
        if bitmask is not None and tuple(bitmask.shape) != (B, (V + 31) // 32):
            raise ValueError("bitmask must be [B, ceil(V/32)]")
        for name, t, dt in (("temperature", temperature, torch.float32),
                            ("top_k", top_k, torch.int32), ("top_p", top_p, torch.float32),
                            ("seed", seed, torch.int64), ("offset", offset, torch.int64)):
            self._check_tensor(t, name, dt)
            if t is not None and t.numel() != B:
                raise ValueError(f"{name} must have B={B} entries")
        params = RowParams(*(None if t is None else t.data_ptr()
                             for t in (temperature, top_k, top_p, seed, offset)))
        return B, V, ld, params

    def set_row_info(self, enable=True, max_batch=4096):
        """Per-row diagnostics {path, band, selection rounds, refinement rounds}."""
        if enable:
            self._row_info = torch.zeros((max_batch, 4), dtype=torch.int32, device=self.device)
            _check(self.lib.smp_set_row_info(self.h, _ptr(self._row_info)), "smp_set_row_info")
        else:
            self._row_info = None
            _check(self.lib.smp_set_row_info(self.h, None), "smp_set_row_info")

    def row_info(self, B):
        return None if self._row_info is None else self._row_info[:B]

    def set_kernel(self, kernel):
        """smp_set_kernel: "board" (default) or "split" (bf16 / fp16 logits)."""
        code = {"board": SMP_KERNEL_BOARD, "split": SMP_KERNEL_SPLIT}[kernel]
        _check(self.lib.smp_set_kernel(self.h, code), "smp_set_kernel")

    def set_wait_limit(self, cycles=0):
        """smp_set_wait_limit: bound on each device wait (SM cycles; 0 = default)."""
        _check(self.lib.smp_set_wait_limit(self.h, int(cycles)), "smp_set_wait_limit")

    def plan(self, dtype, V, B=1):
        out = [ctypes.c_int() for _ in range(4)]
        rc = self.lib.smp_plan(self.h, _DTYPES[dtype], B, V, *[ctypes.byref(o) for o in out])
        _check(rc, "smp_plan")
        return dict(cluster=out[0].value, slice=out[1].value, smem=out[2].value,
                    capacity=out[3].value)

    # -- entry points -------------------------------------------------------------
    def sample(self, logits, temperature, top_k, top_p, seed, offset, bitmask=None, V=None,
               kept_mask=None, kept_count=None, want_mask=False, tokens=None, status=None,
               want_logprob=False, logprobs=None):
        """smp_sample, or smp_sample_logprob when want_logprob or logprobs (float32
        [B]) is given: the log of each drawn token's final probability."""
        B, V, ld, params = self._prep(logits, V, bitmask, temperature, top_k, top_p, seed, offset)
        dev = self.device
        tokens = torch.empty(B, dtype=torch.int32, device=dev) if tokens is None else tokens
        status = torch.empty(B, dtype=torch.int32, device=dev) if status is None else status
        if want_mask and kept_mask is None:
            kept_mask = torch.empty((B, (V + 31) // 32), dtype=torch.int32, device=dev)
            kept_count = torch.empty(B, dtype=torch.int32, device=dev)
        if want_logprob and logprobs is None:
            logprobs = torch.empty(B, dtype=torch.float32, device=dev)
        if logprobs is not None:
            self._check_tensor(logprobs, "logprobs", torch.float32)
            rc = self.lib.smp_sample_logprob(self.h, _ptr(logits), _DTYPES[logits.dtype], B, V,
                                             ld, _ptr(bitmask), ctypes.byref(params),
                                             _ptr(tokens), _ptr(logprobs), _ptr(status),
                                             _ptr(kept_mask), _ptr(kept_count), self._stream())
            _check(rc, "smp_sample_logprob")
        else:
            rc = self.lib.smp_sample(self.h, _ptr(logits), _DTYPES[logits.dtype], B, V, ld,
                                     _ptr(bitmask), ctypes.byref(params), _ptr(tokens),
                                     _ptr(status), _ptr(kept_mask), _ptr(kept_count),
                                     self._stream())
            _check(rc, "smp_sample")
        out = dict(tokens=tokens, status=status, kept_mask=kept_mask, kept_count=kept_count)
        if logprobs is not None:
            out["logprobs"] = logprobs
        return out

    def topk_topp_mask(self, logits, temperature, top_k, top_p, bitmask=None, V=None,
                       want_probs=False):
        B, V, ld, params = self._prep(logits, V, bitmask, temperature, top_k, top_p, None, None)
        dev = self.device
        kept_mask = torch.empty((B, (V + 31) // 32), dtype=torch.int32, device=dev)
        kept_count = torch.empty(B, dtype=torch.int32, device=dev)
        status = torch.empty(B, dtype=torch.int32, device=dev)
        probs = torch.empty((B, V), dtype=torch.float32, device=dev) if want_probs else None
        rc = self.lib.smp_topk_topp_mask(self.h, _ptr(logits), _DTYPES[logits.dtype], B, V, ld,
                                         _ptr(bitmask), ctypes.byref(params), _ptr(kept_mask),
                                         _ptr(kept_count), _ptr(status), _ptr(probs),
                                         self._stream())
        _check(rc, "smp_topk_topp_mask")
        return dict(kept_mask=kept_mask, kept_count=kept_count, status=status, probs=probs)

    def argmax(self, logits, bitmask=None, V=None):
        B, V, ld, _ = self._prep(logits, V, bitmask, None, None, None, None, None)
        dev = self.device
        tokens = torch.empty(B, dtype=torch.int32, device=dev)
        status = torch.empty(B, dtype=torch.int32, device=dev)
        rc = self.lib.smp_argmax(self.h, _ptr(logits), _DTYPES[logits.dtype], B, V, ld,
                                 _ptr(bitmask), _ptr(tokens), _ptr(status), self._stream())
        _check(rc, "smp_argmax")
        return dict(tokens=tokens, status=status)

    def repetition_penalty(self, logits, history, penalty, V=None, status=None):
        """Repetition penalty in place on logits ([B, ld]): history int32 [B, H]
        (entries outside [0, V) are padding), penalty float32 [B].  Returns the
        per-row status tensor."""
        if logits.dtype not in _DTYPES:
            raise ValueError(f"unsupported logits dtype {logits.dtype}")
        self._check_tensor(logits, "logits")
        self._check_tensor(history, "history", torch.int32)
        self._check_tensor(penalty, "penalty", torch.float32)
        B, ld = logits.shape
        V = ld if V is None else V
        if history.dim() != 2 or history.shape[0] != B or penalty.numel() != B:
            raise ValueError("history must be [B, H] and penalty [B]")
        H = history.shape[1]
        status = torch.empty(B, dtype=torch.int32, device=self.device) if status is None \
            else status
        self._check_tensor(status, "status", torch.int32)
        rc = self.lib.smp_repetition_penalty(self.h, _ptr(logits), _DTYPES[logits.dtype], B, V,
                                             ld, _ptr(history) if H else None, H, H,
                                             _ptr(penalty), _ptr(status), self._stream())
        _check(rc, "smp_repetition_penalty")
        return status

    def gumbel_sample(self, logits, temperature, seed, offset, kept_mask=None, V=None,
                      tokens=None, status=None):
        """Gumbel-max draw per row over the kept set (kept_mask int32 [B, W] as
        written by topk_topp_mask, or None for every token)."""
        B, V, ld, _ = self._prep(logits, V, kept_mask, temperature, None, None, seed, offset)
        dev = self.device
        tokens = torch.empty(B, dtype=torch.int32, device=dev) if tokens is None else tokens
        status = torch.empty(B, dtype=torch.int32, device=dev) if status is None else status
        rc = self.lib.smp_gumbel_sample(self.h, _ptr(logits), _DTYPES[logits.dtype], B, V, ld,
                                        _ptr(kept_mask), _ptr(temperature), _ptr(seed),
                                        _ptr(offset), _ptr(tokens), _ptr(status), self._stream())
        _check(rc, "smp_gumbel_sample")
        return dict(tokens=tokens, status=status)

    def top_logprobs(self, logits, temperature, kept_mask, tokens, logprobs, n, V=None):
        """The n most likely kept tokens per row and their logprobs, from the
        outputs of sample(..., want_mask=True, want_logprob=True)."""
        B, V, ld, _ = self._prep(logits, V, kept_mask, temperature, None, None, None, None)
        self._check_tensor(tokens, "tokens", torch.int32)
        self._check_tensor(logprobs, "logprobs", torch.float32)
        if kept_mask is None:
            raise ValueError("kept_mask is required")
        dev = self.device
        ids = torch.empty((B, n), dtype=torch.int32, device=dev)
        lps = torch.empty((B, n), dtype=torch.float32, device=dev)
        rc = self.lib.smp_top_logprobs(self.h, _ptr(logits), _DTYPES[logits.dtype], B, V, ld,
                                       _ptr(kept_mask), _ptr(temperature), _ptr(tokens),
                                       _ptr(logprobs), n, _ptr(ids), _ptr(lps), self._stream())
        _check(rc, "smp_top_logprobs")
        return dict(ids=ids, logprobs=lps)

    def spec_verify(self, target_probs, draft_probs, draft_tokens, seed, offset, V=None,
                    out_tokens=None, n_accepted=None, status=None):
        """Speculative-decoding verification (exact accept / reject rule).

        target_probs: float32 [B, G+1, ld]; draft_probs: float32 [B, G, ld]
        (None when G == 0); draft_tokens: int32 [B, G] (None when G == 0);
        seed, offset: int64 [B] holding uint64 bit patterns.  Returns
        out_tokens int32 [B, G+1], n_accepted int32 [B], status int32 [B].
        """
        self._check_tensor(target_probs, "target_probs", torch.float32)
        B, G1, ld = target_probs.shape
        G = G1 - 1
        V = ld if V is None else V
        if G > 0:
            self._check_tensor(draft_probs, "draft_probs", torch.float32)
            self._check_tensor(draft_tokens, "draft_tokens", torch.int32)
            if tuple(draft_probs.shape) != (B, G, ld) or tuple(draft_tokens.shape) != (B, G):
                raise ValueError("draft_probs must be [B, G, ld] and draft_tokens [B, G]")
        for name, t in (("seed", seed), ("offset", offset)):
            self._check_tensor(t, name, torch.int64)
            if t.numel() != B:
                raise ValueError(f"{name} must have B={B} entries")
        dev = self.device
        if out_tokens is None:
            out_tokens = torch.empty((B, G + 1), dtype=torch.int32, device=dev)
        n_accepted = torch.empty(B, dtype=torch.int32, device=dev) if n_accepted is None \
            else n_accepted
        status = torch.empty(B, dtype=torch.int32, device=dev) if status is None else status
        for name, t in (("out_tokens", out_tokens), ("n_accepted", n_accepted),
                        ("status", status)):
            self._check_tensor(t, name, torch.int32)
        rc = self.lib.smp_spec_verify(self.h, _ptr(target_probs),
                                      _ptr(draft_probs) if G > 0 else None,
                                      _ptr(draft_tokens) if G > 0 else None, B, G, V, ld,
                                      _ptr(seed), _ptr(offset), _ptr(out_tokens),
                                      _ptr(n_accepted), _ptr(status), self._stream())
        _check(rc, "smp_spec_verify")
        return dict(tokens=out_tokens, n_accepted=n_accepted, status=status)


def sample_noalloc(logits, temperature, top_k, top_p, seed, offset, tokens, status,
                   bitmask=None, V=None, kept_mask=None, kept_count=None, lib=None):
    """smp_sample_noalloc: sampling with no handle and no device allocation.

    For callers that may not allocate device memory.  The library allocates
    nothing here, and neither does this wrapper: the caller passes every
    output (tokens, status and, optionally, kept_mask and kept_count).  The
    call runs on the current stream of the device that holds ``logits``.
    Tensor layouts are those of ``Sampler.sample``.
    """
    L = lib or load_library()
    if logits.dtype not in _DTYPES:
        raise ValueError(f"unsupported logits dtype {logits.dtype}")
    dev = logits.device
    ts = (logits, bitmask, temperature, top_k, top_p, seed, offset, tokens, status, kept_mask,
          kept_count)
    for t in ts:
        if t is not None and (not t.is_cuda or t.device != dev or not t.is_contiguous()):
            raise ValueError(f"every tensor must be contiguous and on {dev}")
    B, ld = logits.shape
    V = ld if V is None else V
    params = RowParams(*(t.data_ptr() for t in (temperature, top_k, top_p, seed, offset)))
    with torch.cuda.device(dev):
        stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
        rc = L.smp_sample_noalloc(_ptr(logits), _DTYPES[logits.dtype], B, V, ld, _ptr(bitmask),
                                  ctypes.byref(params), _ptr(tokens), _ptr(status),
                                  _ptr(kept_mask), _ptr(kept_count), stream)
    _check(rc, "smp_sample_noalloc")
    return dict(tokens=tokens, status=status, kept_mask=kept_mask, kept_count=kept_count)
