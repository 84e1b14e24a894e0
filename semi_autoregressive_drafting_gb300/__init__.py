"""libdspark Python binding: DSpark's semi-autoregressive draft-sampling hot path on GB300.

Every function here only marshals arguments: it checks dtypes and devices, allocates the
output tensors with PyTorch (device memory is PyTorch's job) and calls the C ABI declared in
``include/dspark.h``.  All arithmetic runs in the CUDA kernels of ``libdspark.so``; there is no
fallback path, and a missing library raises.

Names follow the pages: B requests, block size gamma, vocab V, Markov rank r, hidden size d,
temperature T; W1 (embedding, [V][r]), W2 (logit projection: [r][V] as the pages write it with
``w2_layout="rv"``, or a linear layer's [V][r] weight with the default ``"vr"``), w (confidence
weight [d + r]), Wj (RNN joint projection [3r][2r + d]), U (base logits [B][gamma][V]),
h (hidden states [B][gamma][d]), x0 (anchors [B]).
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import _lib

__all__ = ["Workspace", "markov_draft", "rnn_draft", "confidence", "tv_label",
           "prefix_schedule", "draft_path", "draft_launches", "draft_loss_launches",
           "DraftOutput", "DraftPlan",
           "VerifyWorkspace", "verify", "LossWorkspace", "draft_loss", "sts", "CapacityRing"]

_F32, _BF16 = 0, 1
_W2_LAYOUT = {"vr": 0, "rv": 1}


def _w2_code(layout: str) -> int:
    if layout not in _W2_LAYOUT:
        raise ValueError(f"w2_layout must be 'vr' ([V][r]) or 'rv' ([r][V]), not {layout!r}")
    return _W2_LAYOUT[layout]


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return _F32
    if t.dtype == torch.bfloat16:
        return _BF16
    raise TypeError(f"unsupported dtype {t.dtype}: use float32 or bfloat16")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libdspark takes device tensors")
    if not t.is_contiguous():
        raise ValueError("libdspark takes contiguous tensors")
    return t.data_ptr()


def _stream(stream) -> int | None:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


class Workspace:
    """Zero-initialised device scratch for the draft calls; reusable across calls of the same
    or smaller shape, one call at a time (stream order)."""

    def __init__(self, head: int, B: int, gamma: int, V: int, r: int, d: int, device=None,
                 target: bool = False, w2_layout: str = "vr"):
        lib = _lib.load()
        flags = (1 if target else 0) | (2 if _w2_code(w2_layout) == 1 else 0)
        n = lib.dspark_workspace_bytes(head, B, gamma, V, r, d, flags)
        if n == 0:
            raise ValueError("invalid draft shape for a workspace")
        self.nbytes = int(n)
        self.buf = torch.zeros(self.nbytes, dtype=torch.uint8, device=device or "cuda")

    def status(self, stream=None) -> int:
        """Synchronise and read (then clear) the device status word."""
        return _lib.load().dspark_get_status(self.buf.data_ptr(), self.nbytes, _stream(stream))


@dataclass
class DraftOutput:
    tokens: torch.Tensor          # [B, gamma] int32
    lse: torch.Tensor             # [B, gamma] fp32, log-sum-exp of (U + B_k) / T
    c: torch.Tensor | None        # [B, gamma] Eq 7 confidence
    S: torch.Tensor | None        # [B, gamma] prefix survival
    cstar: torch.Tensor | None    # [B, gamma] Eq 8 soft acceptance label
    l1: torch.Tensor | None       # [B, gamma] ||p^d - p^t||_1
    logits: torch.Tensor | None   # [B, gamma, V] z = U + B_k (debug)
    s_out: torch.Tensor | None    # [B, r] final RNN state


class DraftPlan:
    """A draft call with its arguments marshalled once: ``run()`` enqueues it again with the
    same input and output buffers (one C call, no per-call allocation or checks)."""

    def __init__(self, head, W1, W2, U, x0, *, T, seed, h, w, Wj, target, forced, s0,
                 want_logits, workspace, stream, out=None, w2_layout="vr"):
        lib = _lib.load()
        B, gamma, V = U.shape
        r = W1.shape[1]
        d = h.shape[2] if h is not None else 0
        dev = U.device
        w2c = _w2_code(w2_layout)
        if tuple(W2.shape) != ((r, V) if w2c == 1 else (V, r)):
            raise ValueError(f"W2 must be {'[r][V]' if w2c == 1 else '[V][r]'} for w2_layout={w2_layout!r}")
        if workspace is None:
            workspace = Workspace(head, B, gamma, V, r, d, device=dev, target=target is not None,
                                  w2_layout=w2_layout)
        f32 = dict(dtype=torch.float32, device=dev)
        o = dict(out or {})
        conf = h is not None and w is not None

        def buf(name, shape, want, dtype=torch.float32):
            if not want:
                return None
            t = o.get(name)
            return t if t is not None else torch.empty(*shape, dtype=dtype, device=dev)

        tokens = buf("tokens", (B, gamma), True, torch.int32)
        lse = buf("lse", (B, gamma), True)
        c = buf("c", (B, gamma), conf)
        S = buf("S", (B, gamma), conf)
        cstar = buf("cstar", (B, gamma), target is not None)
        l1 = buf("l1", (B, gamma), target is not None)
        logits = buf("logits", (B, gamma, V), want_logits)
        s_out = buf("s_out", (B, r), head == 1)
        if x0.dtype != torch.int32 or (forced is not None and forced.dtype != torch.int32):
            raise TypeError("x0 and forced are int32")
        if target is not None and target.dtype != torch.float32:
            raise TypeError("target is float32")
        wdt, udt = _dtype_code(W1), _dtype_code(U)
        for t in (W2, w, Wj):
            if t is not None and _dtype_code(t) != wdt:
                raise TypeError("W1, W2, w and Wj share one dtype")
        if h is not None and _dtype_code(h) != udt:
            raise TypeError("U and h share one dtype")
        common_in = [_ptr(x0), _ptr(forced), _ptr(target)]
        outs = [_ptr(tokens), _ptr(lse), _ptr(c), _ptr(S), _ptr(cstar), _ptr(l1), _ptr(logits)]
        ws = [workspace.buf.data_ptr(), workspace.nbytes, _stream(stream)]
        if head == 0:
            self._fn = lib.dspark_markov_draft
            self._args = (B, gamma, V, r, d, float(T), int(seed), wdt, _ptr(W1), _ptr(W2), w2c,
                          _ptr(w), udt, _ptr(U), _ptr(h), *common_in, *outs, *ws)
            self._where = "dspark_markov_draft"
        else:
            self._fn = lib.dspark_rnn_draft
            self._args = (B, gamma, V, r, d, float(T), int(seed), wdt, _ptr(W1), _ptr(W2), w2c,
                          _ptr(w), _ptr(Wj), udt, _ptr(U), _ptr(h), *common_in, _ptr(s0), *outs,
                          _ptr(s_out), *ws)
            self._where = "dspark_rnn_draft"
        # keep every tensor whose address is baked into the arguments alive
        self._keep = (W1, W2, U, x0, h, w, Wj, target, forced, s0)
        self.workspace = workspace
        self.out = DraftOutput(tokens, lse, c, S, cstar, l1, logits, s_out)

    def run(self, stream=None) -> DraftOutput:
        """Enqueue the call; ``stream`` (a torch stream) overrides the one given at
        construction, e.g. the capturing stream of a CUDA graph."""
        args = self._args if stream is None else self._args[:-1] + (_stream(stream),)
        code = self._fn(*args)
        if code != 0:
            _lib.check(code, self._where)
        return self.out


def _draft(head, W1, W2, U, x0, **kw):
    return DraftPlan(head, W1, W2, U, x0, **kw).run()


def markov_draft(W1, W2, U, x0, *, T=1.0, seed=0, h=None, w=None, target=None, forced=None,
                 want_logits=False, workspace=None, stream=None, out=None,
                 w2_layout="vr") -> DraftOutput:
    """One draft block with the Markov head (Eq 5), sampling, Eq 7 confidence and S_k, and
    the Eq 8 label when ``target`` is given.  ``w2_layout``: "vr" for W2 [V][r], "rv" for
    [r][V].  See ``dspark_markov_draft``."""
    return _draft(0, W1, W2, U, x0, T=T, seed=seed, h=h, w=w, Wj=None, target=target,
                  forced=forced, s0=None, want_logits=want_logits, workspace=workspace,
                  stream=stream, out=out, w2_layout=w2_layout)


def rnn_draft(W1, W2, Wj, U, h, x0, *, T=1.0, seed=0, w=None, target=None, forced=None, s0=None,
              want_logits=False, workspace=None, stream=None, out=None,
              w2_layout="vr") -> DraftOutput:
    """One draft block with the RNN head (Eq 6).  See ``dspark_rnn_draft``."""
    return _draft(1, W1, W2, U, x0, T=T, seed=seed, h=h, w=w, Wj=Wj, target=target,
                  forced=forced, s0=s0, want_logits=want_logits, workspace=workspace,
                  stream=stream, out=out, w2_layout=w2_layout)


def confidence(W1, w, h, x0, tokens, *, stream=None):
    """Teacher-forced Eq 7 confidence and prefix survival for given tokens."""
    lib = _lib.load()
    B, gamma, d = h.shape
    V, r = W1.shape
    c = torch.empty(B, gamma, dtype=torch.float32, device=h.device)
    S = torch.empty_like(c)
    code = lib.dspark_confidence(B, gamma, V, r, d, _dtype_code(W1), _ptr(W1), _ptr(w),
                                 _dtype_code(h), _ptr(h), _ptr(x0), _ptr(tokens), _ptr(c),
                                 _ptr(S), _stream(stream))
    _lib.check(code, "dspark_confidence")
    return c, S


def tv_label(draft_logits, target_logits, *, T=1.0, stream=None):
    """Eq 8 soft acceptance label c* and the L1 distance on [N, V] fp32 logit rows."""
    lib = _lib.load()
    N, V = draft_logits.shape
    cstar = torch.empty(N, dtype=torch.float32, device=draft_logits.device)
    l1 = torch.empty_like(cstar)
    code = lib.dspark_tv_label(N, V, float(T), _ptr(draft_logits), _ptr(target_logits),
                               _ptr(cstar), _ptr(l1), _stream(stream))
    _lib.check(code, "dspark_tv_label")
    return cstar, l1


def prefix_schedule(S, sps, *, stream=None, out=None):
    """Per-request verify lengths maximising SPS(n) * expected accepted tokens.

    ``out``: optional preallocated (lengths [B] int32, theta [1] float64) device tensors, e.g.
    to capture the call in a CUDA graph."""
    lib = _lib.load()
    B, gamma = S.shape
    if out is not None:
        ln, theta = out
    else:
        ln = torch.empty(B, dtype=torch.int32, device=S.device)
        theta = torch.empty(1, dtype=torch.float64, device=S.device)
    code = lib.dspark_prefix_schedule(B, gamma, _ptr(S), _ptr(sps), _ptr(ln), _ptr(theta),
                                      _stream(stream))
    _lib.check(code, "dspark_prefix_schedule")
    return ln, theta


class VerifyWorkspace(Workspace):
    """Zero-initialised device scratch for ``verify`` (shapes up to B, gamma, V)."""

    def __init__(self, B: int, gamma: int, V: int, device=None):
        n = _lib.load().dspark_verify_workspace_bytes(B, gamma, V)
        if n == 0:
            raise ValueError("invalid verify shape for a workspace")
        self.nbytes = int(n)
        self.buf = torch.zeros(self.nbytes, dtype=torch.uint8, device=device or "cuda")


def verify(draft_logits, target_logits, draft_tokens, *, T=1.0, seed=0, workspace=None,
           stream=None, out=None):
    """Speculative accept/reject of one draft block per request.  See ``dspark_verify``.

    draft_logits [B, gamma, V] fp32, target_logits [B, gamma + 1, V] fp32, draft_tokens
    [B, gamma] int32.  Returns (n_accepted [B] int32, out_tokens [B, gamma + 1] int32).
    """
    lib = _lib.load()
    B, gamma, V = draft_logits.shape
    if draft_logits.dtype != torch.float32 or target_logits.dtype != torch.float32:
        raise TypeError("verify takes fp32 logits")
    if tuple(target_logits.shape) != (B, gamma + 1, V) or tuple(draft_tokens.shape) != (B, gamma):
        raise ValueError("target_logits must be [B, gamma + 1, V] and draft_tokens [B, gamma]")
    ws = workspace or VerifyWorkspace(B, gamma, V, device=draft_logits.device)
    if out is None:
        n = torch.empty(B, dtype=torch.int32, device=draft_logits.device)
        toks = torch.empty(B, gamma + 1, dtype=torch.int32, device=draft_logits.device)
    else:
        n, toks = out
    code = lib.dspark_verify(B, gamma, V, float(T), int(seed) & (2**64 - 1), _ptr(draft_logits),
                             _ptr(target_logits), _ptr(draft_tokens), _ptr(n), _ptr(toks),
                             ws.buf.data_ptr(), ws.nbytes, _stream(stream))
    _lib.check(code, "dspark_verify")
    return n, toks


class LossWorkspace(Workspace):
    """Device scratch for ``draft_loss`` (shapes up to B, gamma, V)."""

    def __init__(self, B: int, gamma: int, V: int, device=None):
        n = _lib.load().dspark_draft_loss_workspace_bytes(B, gamma, V)
        if n == 0:
            raise ValueError("invalid loss shape for a workspace")
        self.nbytes = int(n)
        self.buf = torch.zeros(self.nbytes, dtype=torch.uint8, device=device or "cuda")


def draft_loss(draft_logits, target_logits, labels, conf_logits, *, T=1.0,
               alpha=(0.1, 0.9, 1.0), want_grads=True, workspace=None, stream=None):
    """Eqs 9-12 and their gradients (c* held as a label).  See ``dspark_draft_loss``.

    Returns (loss [B], parts [B, 3], grad_logits [B, gamma, V] or None, grad_conf [B, gamma]
    or None), all fp32.
    """
    lib = _lib.load()
    B, gamma, V = draft_logits.shape
    if draft_logits.dtype != torch.float32 or target_logits.dtype != torch.float32:
        raise TypeError("draft_loss takes fp32 logits")
    dev = draft_logits.device
    ws = workspace or LossWorkspace(B, gamma, V, device=dev)
    loss = torch.empty(B, dtype=torch.float32, device=dev)
    parts = torch.empty(B, 3, dtype=torch.float32, device=dev)
    gz = torch.empty_like(draft_logits) if want_grads else None
    gc = torch.empty(B, gamma, dtype=torch.float32, device=dev) if want_grads else None
    code = lib.dspark_draft_loss(B, gamma, V, float(T), _ptr(draft_logits), _ptr(target_logits),
                                 _ptr(labels), _ptr(conf_logits), float(alpha[0]),
                                 float(alpha[1]), float(alpha[2]), _ptr(loss), _ptr(parts),
                                 _ptr(gz), _ptr(gc), ws.buf.data_ptr(), ws.nbytes, _stream(stream))
    _lib.check(code, "dspark_draft_loss")
    return loss, parts, gz, gc


def sts(conf_logits, accepted, grid, *, bins=15, stream=None):
    """Sequential temperature scaling of the confidence head.  See ``dspark_sts``.

    conf_logits [N, gamma] fp32, accepted [N] int32, grid [ngrid] fp32.  Returns (tau [gamma],
    ece [gamma], ece_grid [gamma, ngrid]) fp32 and the device status.
    """
    lib = _lib.load()
    N, gamma = conf_logits.shape
    ng = grid.shape[0]
    n = lib.dspark_sts_workspace_bytes(N, gamma, ng, bins)
    if n == 0:
        raise ValueError("invalid sts shape")
    ws = Workspace.__new__(Workspace)
    ws.nbytes = int(n)
    ws.buf = torch.zeros(ws.nbytes, dtype=torch.uint8, device=conf_logits.device)
    tau = torch.empty(gamma, dtype=torch.float32, device=conf_logits.device)
    ece = torch.empty_like(tau)
    eg = torch.empty(gamma, ng, dtype=torch.float32, device=conf_logits.device)
    code = lib.dspark_sts(N, gamma, _ptr(conf_logits), _ptr(accepted), ng, _ptr(grid), bins,
                          _ptr(tau), _ptr(ece), _ptr(eg), ws.buf.data_ptr(), ws.nbytes,
                          _stream(stream))
    _lib.check(code, "dspark_sts")
    return tau, ece, eg, ws.status(stream)


class CapacityRing:
    """The steps/s table the prefix scheduler reads, delayed by ``delay`` steps.

    "DSpark：既要猜得连贯…" ("设计") notes that the production scheduler uses a capacity
    estimate delayed by two steps, to fit asynchronous scheduling and CUDA Graphs.  ``table`` is
    one fixed device buffer that ``prefix_schedule`` can read (also from a captured graph);
    ``advance(sps)`` records this step's measured table and copies the one recorded ``delay``
    steps earlier into ``table``, stream-ordered (until ``delay`` steps have been recorded,
    ``table`` keeps the initial table).  Only tensor copies: no arithmetic of the method here.
    """

    def __init__(self, initial, delay: int = 2):
        if delay < 0:
            raise ValueError("delay must be >= 0")
        self.delay = delay
        self.table = initial.clone()
        self._ring = [torch.empty_like(initial) for _ in range(delay + 1)]
        self._step = 0

    def advance(self, sps) -> "torch.Tensor":
        slot = self._step % (self.delay + 1)
        self._ring[slot].copy_(sps, non_blocking=True)
        if self._step >= self.delay:
            self.table.copy_(self._ring[(self._step - self.delay) % (self.delay + 1)], non_blocking=True)
        self._step += 1
        return self.table


def draft_path(head: int, B: int, V: int, r: int, bf16: bool = True) -> int:
    return _lib.load().dspark_draft_path(head, B, V, r, _BF16 if bf16 else _F32)


def draft_launches(head: int, B: int, V: int, r: int, bf16: bool = True) -> int:
    return _lib.load().dspark_draft_launches(head, B, V, r, _BF16 if bf16 else _F32)


def draft_cluster(head: int, B: int, V: int, r: int, bf16: bool = True) -> int:
    """Blocks per thread-block cluster of the draft kernel these arguments select (1: none)."""
    return _lib.load().dspark_draft_cluster(head, B, V, r, _BF16 if bf16 else _F32)


def draft_loss_launches(B: int, gamma: int, V: int, with_grad: bool = True) -> int:
    """Kernel launches of one draft_loss call (the sub-batch pipeline and the totals)."""
    return _lib.load().dspark_draft_loss_launches(B, gamma, V, int(with_grad))
