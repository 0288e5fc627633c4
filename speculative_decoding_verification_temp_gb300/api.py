"""Thin torch binding over the C ABI: argument marshalling only.

Every step of the verification runs inside libspecverify.so on the GPU; this
module checks tensor placement and layout, allocates the outputs, and passes
raw device pointers and torch's current CUDA stream to the C functions.
"""

import ctypes
from collections import namedtuple

import torch

from . import _abi

ChainResult = namedtuple("ChainResult", "num_accepted tokens flags residual")
TreeResult = namedtuple("TreeResult", "num_accepted path tokens flags residual")
MaskResult = namedtuple("MaskResult", "mask position flags")

_DTYPES = {torch.float32: _abi.SPEC_F32, torch.bfloat16: _abi.SPEC_BF16}


class SpecVerifyError(RuntimeError):
    """A non-OK status returned by the C ABI."""


def _check(code):
    if code != _abi.SPEC_OK:
        raise SpecVerifyError(_abi.status_string(code))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def set_wait_limit(cycles=None):
    """spec_set_wait_limit: bound the streaming chain path's first wait on each
    chunk to `cycles` SM clock cycles (0: one non-blocking test); None restores
    the default bound.  A wait that gives up turns the call's outputs into the
    documented fallback with FLAG_TIMEOUT (diagnostics and tests)."""
    _check(_abi.load().spec_set_wait_limit(-1 if cycles is None else int(cycles)))


_WORKSPACES = {}


def workspace(device, nbytes):
    """A device workspace of at least nbytes, cached per (device, stream).

    The library needs no initialised workspace: every call first clears the
    part it relies on, so the cached buffer serves successive calls on one
    stream.  Calls on different streams may run concurrently on the GPU, so
    each stream gets a buffer of its own (allocated on that stream).
    """
    dev = torch.device(device)
    index = dev.index if dev.index is not None else torch.cuda.current_device()
    stream = torch.cuda.current_stream(index)
    key = (index, stream.cuda_stream)
    ws = _WORKSPACES.get(key)
    if ws is None or ws.numel() < nbytes:
        with torch.cuda.stream(stream):
            ws = torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=torch.device("cuda", index))
        _WORKSPACES[key] = ws
    return ws


def _top_k(x, n, V, name, device):
    """A per-sequence top-k argument as a device array, or None when no row
    filters.  A host value (scalar, list, numpy array, CPU tensor) whose
    entries are all off (k <= 0 or k >= V) becomes None, so that it does not
    send the call down the top-k path; a CUDA tensor is passed as given."""
    if x is None:
        return None
    if not (isinstance(x, torch.Tensor) and x.is_cuda):
        k = torch.as_tensor(x).to(torch.int64).flatten()
        if not bool(((k > 0) & (k < V)).any()):
            return None
    return _vec(x, n, torch.int32, name, device)


def _rows(x, name):
    """x viewed as rows with one uniform row stride over all leading dims."""
    if x.dim() < 2:
        raise ValueError(f"{name} must have a vocabulary dimension")
    if x.stride(-1) != 1:
        x = x.contiguous()
    ld = x.stride(-2)
    if ld < x.shape[-1]:
        x = x.contiguous()
        ld = x.shape[-1]
    expect = ld
    for d in range(x.dim() - 2, 0, -1):
        expect *= x.shape[d]
        if x.shape[d - 1] > 1 and x.stride(d - 1) != expect:
            x = x.contiguous()
            ld = x.shape[-1]
            break
    return x, ld


def _filter(x, n, name, device, off):
    """A per-sequence top-p or min-p argument as a device float array, or None
    when no row filters: a host value whose entries are all off (off(value)
    true) becomes None; a CUDA tensor is passed as given."""
    if x is None:
        return None
    if not (isinstance(x, torch.Tensor) and x.is_cuda):
        v = torch.as_tensor(x, dtype=torch.float64).flatten()
        if bool(off(v).all()):
            return None
    return _vec(x, n, torch.float32, name, device)


def _topp_off(v):
    return ~(v < 1.0)  # >= 1 or NaN


def _minp_off(v):
    return ~(v > 0.0)  # <= 0 or NaN


def _policy(temperature, top_k, top_p, min_p):
    """A spec_policy over device arrays (top_k, top_p and min_p may be None)."""
    ptr = lambda t: None if t is None else t.data_ptr()
    return _abi.spec_policy(temperature.data_ptr(), ptr(top_k), ptr(top_p), ptr(min_p))


def _vec(x, n, dtype, name, device):
    t = torch.as_tensor(x, device=device)
    if t.dim() == 0:
        t = t.expand(n)
    t = t.to(dtype).contiguous()
    if t.numel() != n:
        raise ValueError(f"{name} must hold {n} values")
    return t


def _cuda_tensor(x, name):
    if not isinstance(x, torch.Tensor) or not x.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    return x


def verify_chain(target_logits, draft_logits, draft_tokens, target_temperature,
                 draft_temperature, target_top_k=None, draft_top_k=None, seed=0,
                 uniform_override=None, return_residual=False, workspace_tensor=None,
                 target_top_p=None, draft_top_p=None, target_min_p=None, draft_min_p=None):
    """Chain speculative-sampling verification on the GPU (see spec_verify_chain).

    target_logits [B, gamma+1, V] and draft_logits [B, gamma, V] (float32 or
    bfloat16, CUDA), draft_tokens [B, gamma] integer; temperatures and top-k
    per sequence (scalars broadcast).  Returns ChainResult with
    num_accepted [B] int32, tokens [B, gamma+1] int32, flags [B] int32 (bit
    pattern of the SPEC_FLAG_* values) and residual [B, V] float32 or None.
    """
    _cuda_tensor(target_logits, "target_logits")
    dev = target_logits.device
    if target_logits.dtype not in _DTYPES:
        raise ValueError("logits must be float32 or bfloat16")
    B, G1, V = target_logits.shape
    gamma = G1 - 1
    tl, ld_t = _rows(target_logits, "target_logits")
    if gamma > 0:
        _cuda_tensor(draft_logits, "draft_logits")
        if draft_logits.dtype != target_logits.dtype or tuple(draft_logits.shape) != (B, gamma, V):
            raise ValueError("draft_logits must be [B, gamma, V] with the target's dtype")
        dl, ld_d = _rows(draft_logits, "draft_logits")
        toks = _vec(draft_tokens, B * gamma, torch.int32, "draft_tokens", dev).view(B, gamma)
    else:
        dl, ld_d, toks = None, 0, None
    tp = _vec(target_temperature, B, torch.float32, "target_temperature", dev)
    tq = _vec(draft_temperature, B, torch.float32, "draft_temperature", dev)
    kp = _top_k(target_top_k, B, V, "target_top_k", dev)
    kq = _top_k(draft_top_k, B, V, "draft_top_k", dev)
    pp = _filter(target_top_p, B, "target_top_p", dev, _topp_off)
    pq = _filter(draft_top_p, B, "draft_top_p", dev, _topp_off)
    mp = _filter(target_min_p, B, "target_min_p", dev, _minp_off)
    mq = _filter(draft_min_p, B, "draft_min_p", dev, _minp_off)
    uov = None
    if uniform_override is not None:
        uov = _vec(uniform_override, B * G1 * 2, torch.float32, "uniform_override", dev)
    num = torch.empty(B, dtype=torch.int32, device=dev)
    out = torch.empty((B, G1), dtype=torch.int32, device=dev)
    flags = torch.empty(B, dtype=torch.int32, device=dev)
    resid = torch.empty((B, V), dtype=torch.float32, device=dev) if return_residual else None
    lib = _abi.load()
    dt = _DTYPES[target_logits.dtype]
    nbytes = lib.spec_verify_chain_workspace_size(B, gamma, V, dt)
    ws = workspace(dev, nbytes) if workspace_tensor is None else workspace_tensor
    code = lib.spec_verify_chain(
        _ptr(tl), ld_t, _ptr(dl), ld_d, dt, B, gamma, V, _ptr(toks),
        _policy(tp, kp, pp, mp),
        _policy(tq, kq, pq, mq),
        int(seed) & ((1 << 64) - 1), _ptr(uov), _ptr(num), _ptr(out), _ptr(flags), _ptr(resid),
        _ptr(ws), ws.numel(), _stream(dev))
    _check(code)
    return ChainResult(num, out, flags, resid)


def verify_tree(target_logits, draft_logits, node_tokens, parent, max_depth,
                target_temperature, draft_temperature, target_top_k=None, draft_top_k=None,
                seed=0, uniform_override=None, return_residual=False, workspace_tensor=None,
                target_top_p=None, draft_top_p=None, target_min_p=None, draft_min_p=None):
    """Tree verification by recursive rejection on the GPU (see spec_verify_tree).

    target_logits, draft_logits [T, N, V]; node_tokens, parent [T, N].
    Returns TreeResult with num_accepted [T], path and tokens [T, max_depth+1],
    flags [T] and residual [T, V] or None.
    """
    _cuda_tensor(target_logits, "target_logits")
    _cuda_tensor(draft_logits, "draft_logits")
    dev = target_logits.device
    if target_logits.dtype not in _DTYPES or draft_logits.dtype != target_logits.dtype:
        raise ValueError("logits must both be float32 or both bfloat16")
    T, N, V = target_logits.shape
    if tuple(draft_logits.shape) != (T, N, V):
        raise ValueError("draft_logits must be [T, N, V]")
    tl, ld_t = _rows(target_logits, "target_logits")
    dl, ld_d = _rows(draft_logits, "draft_logits")
    toks = _vec(node_tokens, T * N, torch.int32, "node_tokens", dev)
    par = _vec(parent, T * N, torch.int32, "parent", dev)
    tp = _vec(target_temperature, T, torch.float32, "target_temperature", dev)
    tq = _vec(draft_temperature, T, torch.float32, "draft_temperature", dev)
    kp = _top_k(target_top_k, T, V, "target_top_k", dev)
    kq = _top_k(draft_top_k, T, V, "draft_top_k", dev)
    pp = _filter(target_top_p, T, "target_top_p", dev, _topp_off)
    pq = _filter(draft_top_p, T, "draft_top_p", dev, _topp_off)
    mp = _filter(target_min_p, T, "target_min_p", dev, _minp_off)
    mq = _filter(draft_min_p, T, "draft_min_p", dev, _minp_off)
    uov = None
    if uniform_override is not None:
        uov = _vec(uniform_override, T * N * 2, torch.float32, "uniform_override", dev)
    W = int(max_depth) + 1
    num = torch.empty(T, dtype=torch.int32, device=dev)
    path = torch.empty((T, W), dtype=torch.int32, device=dev)
    out = torch.empty((T, W), dtype=torch.int32, device=dev)
    flags = torch.empty(T, dtype=torch.int32, device=dev)
    resid = torch.empty((T, V), dtype=torch.float32, device=dev) if return_residual else None
    lib = _abi.load()
    dt = _DTYPES[target_logits.dtype]
    nbytes = lib.spec_verify_tree_workspace_size(T, N, V, dt)
    ws = workspace(dev, nbytes) if workspace_tensor is None else workspace_tensor
    code = lib.spec_verify_tree(
        _ptr(tl), ld_t, _ptr(dl), ld_d, dt, T, N, V, int(max_depth), _ptr(toks), _ptr(par),
        _policy(tp, kp, pp, mp),
        _policy(tq, kq, pq, mq),
        int(seed) & ((1 << 64) - 1), _ptr(uov), _ptr(num), _ptr(path), _ptr(out), _ptr(flags),
        _ptr(resid), _ptr(ws), ws.numel(), _stream(dev))
    _check(code)
    return TreeResult(num, path, out, flags, resid)


def verify_chain_static(target_logits, draft_logits, draft_tokens, target_temperature,
                        draft_temperature, target_top_k=None, draft_top_k=None, seed=0,
                        uniform_override=None, return_residual=False, target_top_p=None,
                        draft_top_p=None, target_min_p=None, draft_min_p=None):
    """verify_chain on the library's fixed scratch (see spec_verify_chain_static).

    Same arguments and result as verify_chain, without a workspace: the C call
    allocates nothing (this wrapper still allocates the output tensors).  Calls
    on one device must not overlap on the GPU; shapes whose workspace exceeds
    SPEC_STATIC_SCRATCH_BYTES raise SpecVerifyError (SPEC_ERR_UNSUPPORTED).
    """
    _cuda_tensor(target_logits, "target_logits")
    dev = target_logits.device
    if target_logits.dtype not in _DTYPES:
        raise ValueError("logits must be float32 or bfloat16")
    B, G1, V = target_logits.shape
    gamma = G1 - 1
    tl, ld_t = _rows(target_logits, "target_logits")
    if gamma > 0:
        _cuda_tensor(draft_logits, "draft_logits")
        if draft_logits.dtype != target_logits.dtype or tuple(draft_logits.shape) != (B, gamma, V):
            raise ValueError("draft_logits must be [B, gamma, V] with the target's dtype")
        dl, ld_d = _rows(draft_logits, "draft_logits")
        toks = _vec(draft_tokens, B * gamma, torch.int32, "draft_tokens", dev).view(B, gamma)
    else:
        dl, ld_d, toks = None, 0, None
    tp = _vec(target_temperature, B, torch.float32, "target_temperature", dev)
    tq = _vec(draft_temperature, B, torch.float32, "draft_temperature", dev)
    kp = _top_k(target_top_k, B, V, "target_top_k", dev)
    kq = _top_k(draft_top_k, B, V, "draft_top_k", dev)
    pp = _filter(target_top_p, B, "target_top_p", dev, _topp_off)
    pq = _filter(draft_top_p, B, "draft_top_p", dev, _topp_off)
    mp = _filter(target_min_p, B, "target_min_p", dev, _minp_off)
    mq = _filter(draft_min_p, B, "draft_min_p", dev, _minp_off)
    uov = None
    if uniform_override is not None:
        uov = _vec(uniform_override, B * G1 * 2, torch.float32, "uniform_override", dev)
    num = torch.empty(B, dtype=torch.int32, device=dev)
    out = torch.empty((B, G1), dtype=torch.int32, device=dev)
    flags = torch.empty(B, dtype=torch.int32, device=dev)
    resid = torch.empty((B, V), dtype=torch.float32, device=dev) if return_residual else None
    lib = _abi.load()
    with torch.cuda.device(dev):
        code = lib.spec_verify_chain_static(
            _ptr(tl), ld_t, _ptr(dl), ld_d, _DTYPES[target_logits.dtype], B, gamma, V,
            _ptr(toks),
            _policy(tp, kp, pp, mp),
            _policy(tq, kq, pq, mq),
            int(seed) & ((1 << 64) - 1), _ptr(uov), _ptr(num), _ptr(out), _ptr(flags),
            _ptr(resid), _stream(dev))
    _check(code)
    return ChainResult(num, out, flags, resid)


def tree_mask(parent, max_depth):
    """Ancestor-or-self masks and depth positions (see spec_tree_mask).

    parent [T, N] (CUDA).  Returns MaskResult with mask [T, N, ceil(N/64)]
    int64 (the uint64 bit words), position [T, N] int32, flags [T] int32.
    """
    _cuda_tensor(parent, "parent")
    dev = parent.device
    T, N = parent.shape
    par = parent.to(torch.int32).contiguous()
    words = (N + 63) // 64
    mask = torch.empty((T, N, words), dtype=torch.int64, device=dev)
    pos = torch.empty((T, N), dtype=torch.int32, device=dev)
    flags = torch.empty(T, dtype=torch.int32, device=dev)
    code = _abi.load().spec_tree_mask(_ptr(par), T, N, int(max_depth), _ptr(mask), _ptr(pos),
                                      _ptr(flags), _stream(dev))
    _check(code)
    return MaskResult(mask, pos, flags)


OverlapResult = namedtuple("OverlapResult", "beta flags")


def overlap(target_logits, draft_logits, target_temperature, draft_temperature):
    """Per-position overlap beta_i = sum_v min(p_i(v), q_i(v)) (see spec_overlap).

    target_logits [B, gamma+1, V] and draft_logits [B, gamma, V] (float32 or
    bfloat16, CUDA); temperatures per sequence (scalars broadcast).  Returns
    OverlapResult with beta [B, gamma] float32 and flags [B] int32.
    """
    _cuda_tensor(target_logits, "target_logits")
    _cuda_tensor(draft_logits, "draft_logits")
    dev = target_logits.device
    if target_logits.dtype not in _DTYPES or draft_logits.dtype != target_logits.dtype:
        raise ValueError("logits must both be float32 or both bfloat16")
    B, G1, V = target_logits.shape
    gamma = G1 - 1
    if tuple(draft_logits.shape) != (B, gamma, V):
        raise ValueError("draft_logits must be [B, gamma, V]")
    tl, ld_t = _rows(target_logits, "target_logits")
    dl, ld_d = _rows(draft_logits, "draft_logits")
    tp = _vec(target_temperature, B, torch.float32, "target_temperature", dev)
    tq = _vec(draft_temperature, B, torch.float32, "draft_temperature", dev)
    beta = torch.empty((B, gamma), dtype=torch.float32, device=dev)
    flags = torch.empty(B, dtype=torch.int32, device=dev)
    lib = _abi.load()
    code = lib.spec_overlap(_ptr(tl), ld_t, _ptr(dl), ld_d, _DTYPES[target_logits.dtype], B,
                            gamma, V, _abi.spec_policy(tp.data_ptr(), None),
                            _abi.spec_policy(tq.data_ptr(), None), _ptr(beta), _ptr(flags),
                            _stream(dev))
    _check(code)
    return OverlapResult(beta, flags)


TypicalResult = namedtuple("TypicalResult", "num_accepted tokens flags")


def typical_accept(target_logits, draft_tokens, target_temperature, epsilon, delta,
                   workspace_tensor=None):
    """Typical acceptance (see spec_typical_accept): an approximate rule, not
    distribution-exact.

    target_logits [B, gamma+1, V] (float32 or bfloat16, CUDA), draft_tokens
    [B, gamma] integer, temperatures per sequence (scalars broadcast), epsilon
    and delta floats.  Returns TypicalResult with num_accepted [B] int32,
    tokens [B, gamma+1] int32 (-1 padded) and flags [B] int32.
    """
    _cuda_tensor(target_logits, "target_logits")
    dev = target_logits.device
    if target_logits.dtype not in _DTYPES:
        raise ValueError("target_logits must be float32 or bfloat16")
    B, G1, V = target_logits.shape
    gamma = G1 - 1
    tl, ld_t = _rows(target_logits, "target_logits")
    toks = None
    if gamma > 0:
        toks = _vec(draft_tokens, B * gamma, torch.int32, "draft_tokens", dev).view(B, gamma)
    tp = _vec(target_temperature, B, torch.float32, "target_temperature", dev)
    num = torch.empty(B, dtype=torch.int32, device=dev)
    out = torch.empty((B, G1), dtype=torch.int32, device=dev)
    flags = torch.empty(B, dtype=torch.int32, device=dev)
    lib = _abi.load()
    nbytes = lib.spec_typical_workspace_size(B, gamma, V, _DTYPES[target_logits.dtype])
    ws = workspace(dev, nbytes) if workspace_tensor is None else workspace_tensor
    code = lib.spec_typical_accept(_ptr(tl), ld_t, _DTYPES[target_logits.dtype], B, gamma, V,
                                   _abi.spec_policy(tp.data_ptr(), None),
                                   None if toks is None else _ptr(toks), float(epsilon),
                                   float(delta), _ptr(num), _ptr(out), _ptr(flags), _ptr(ws),
                                   ws.numel(), _stream(dev))
    _check(code)
    return TypicalResult(num, out, flags)


RerankResult = namedtuple("RerankResult", "nodes parent value count flags")


def tree_rerank(parent, confidence, m):
    """EAGLE-2 rerank (see spec_tree_rerank): the m nodes of highest path
    product of confidences per tree, ascending, with re-indexed parents.

    parent [T, N] integer and confidence [T, N] float (CUDA tensors or
    arrays).  Returns RerankResult with nodes, parent [T, m] int32, value
    [T, m] float32, count [T] int32 and flags [T] int32.
    """
    par = torch.as_tensor(parent)
    if par.dim() == 1:
        par = par.unsqueeze(0)
    T, N = par.shape
    dev = par.device if par.is_cuda else torch.device("cuda", torch.cuda.current_device())
    par = par.to(device=dev, dtype=torch.int32).contiguous()
    conf = torch.as_tensor(confidence).to(device=dev, dtype=torch.float32).reshape(T, N).contiguous()
    m = int(m)
    nodes = torch.empty((T, max(m, 1)), dtype=torch.int32, device=dev)
    newp = torch.empty_like(nodes)
    value = torch.empty((T, max(m, 1)), dtype=torch.float32, device=dev)
    count = torch.empty(T, dtype=torch.int32, device=dev)
    flags = torch.empty(T, dtype=torch.int32, device=dev)
    code = _abi.load().spec_tree_rerank(_ptr(par), _ptr(conf), T, N, m, _ptr(nodes), _ptr(newp),
                                        _ptr(value), _ptr(count), _ptr(flags), _stream(dev))
    _check(code)
    return RerankResult(nodes, newp, value, count, flags)
