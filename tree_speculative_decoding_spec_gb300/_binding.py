"""ctypes binding of libspec_tree.so: argument marshalling only.

Every function here takes torch tensors, checks their dtype/shape/device,
allocates outputs and workspace with torch (device memory is plumbing), and
calls the C entry point of the same name; all arithmetic runs in the library's
CUDA kernels.  There is no CPU fallback: if the library is missing, importing
this module raises.
"""

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libspec_tree.so")

SPEC_MAX_T = 1024
SPEC_MAX_DEPTH = 16
SPEC_MAX_TOPK = 16
SPEC_F32, SPEC_BF16 = 0, 1
STATUS_NAMES = {0: "SPEC_OK", 1: "SPEC_EINVAL", 2: "SPEC_ETREE", 3: "SPEC_EALIGN", 4: "SPEC_EWORKSPACE",
                5: "SPEC_EUNSUPPORTED", 6: "SPEC_ECUDA", 7: "SPEC_ETIMEOUT"}

_i32p = ctypes.POINTER(ctypes.c_int32)


class spec_tree(ctypes.Structure):
    _fields_ = [
        ("T", ctypes.c_int32), ("max_depth", ctypes.c_int32), ("words", ctypes.c_int32),
        ("n_internal", ctypes.c_int32),
        ("n_at_depth", ctypes.c_int32 * (SPEC_MAX_DEPTH + 1)),
        ("n_internal_at_depth", ctypes.c_int32 * (SPEC_MAX_DEPTH + 1)),
        ("max_rank_at_depth", ctypes.c_int32 * (SPEC_MAX_DEPTH + 1)),
        ("parent", ctypes.c_void_p), ("depth", ctypes.c_void_p), ("rank", ctypes.c_void_p),
        ("anc", ctypes.c_void_p), ("internal", ctypes.c_void_p), ("internal_off", ctypes.c_void_p),
        ("row_of", ctypes.c_void_p), ("child_off", ctypes.c_void_p), ("child_idx", ctypes.c_void_p),
    ]


class spec_head(ctypes.Structure):
    _fields_ = [("cond", ctypes.c_int32), ("topk", ctypes.c_int32), ("form", ctypes.c_int32), ("hidden", ctypes.c_int32),
                ("W1", ctypes.c_void_p), ("b1", ctypes.c_void_p), ("W1b", ctypes.c_void_p), ("b1b", ctypes.c_void_p),
                ("gamma", ctypes.c_void_p), ("beta", ctypes.c_void_p), ("W2", ctypes.c_void_p)]


class spec_trace_entry(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 48), ("launches", ctypes.c_int32), ("total_ms", ctypes.c_double)]


class SpecError(RuntimeError):
    def __init__(self, fn, status, message):
        self.status = status
        super().__init__(f"{fn} failed with {STATUS_NAMES.get(status, status)}: {message}")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built (run __graft_entry__.build() or python -m "
                          "tree_speculative_decoding_spec_gb300.build)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, sz, i32, u64, f32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.c_uint64, ctypes.c_float
    tp = ctypes.POINTER(spec_tree)
    sig = {
        "spec_tree_device_bytes": (sz, [i32]),
        "spec_tree_build": (i32, [vp, vp, i32, vp, sz, tp, vp]),
        "hydra_draft_workspace_size": (sz, [tp, i32, i32, i32, i32, vp, vp, i32]),
        "hydra_draft": (i32, [vp, vp, i32, vp, vp, vp, vp, vp, vp, tp, i32, i32, i32, i32, vp, vp, vp, vp, sz, vp]),
        "hydra_draft_folded": (i32, [vp, vp, i32, vp, vp, vp, vp, vp, vp, vp, tp, i32, i32, i32, i32, vp, vp, vp, vp, sz,
                                     vp]),
        "hydra_fold_table_bytes": (sz, [i32, i32]),
        "hydra_fold_embedding": (i32, [vp, vp, i32, i32, i32, vp, vp]),
        "hydra_draft_heads_workspace_size": (sz, [tp, i32, i32, i32, i32, ctypes.POINTER(spec_head), i32]),
        "hydra_draft_heads": (i32, [vp, vp, i32, ctypes.POINTER(spec_head), vp, tp, i32, i32, i32, f32, i32, vp, vp,
                                    vp, vp, sz, vp]),
        "tree_attention_workspace_size": (sz, [tp, i32, i32, i32, i32, i32, i32]),
        "tree_attention": (i32, [vp, vp, vp, vp, vp, vp, tp, i32, i32, i32, i32, i32, f32, i32, vp, vp, vp, sz, vp]),
        "tree_attention_noalloc": (i32, [vp, vp, vp, vp, vp, vp, tp, i32, i32, i32, i32, i32, f32, i32, vp, vp, vp]),
        "tree_attention_noalloc_status": (i32, [_i32p, vp]),
        "tree_attention_paged_workspace_size": (sz, [tp, i32, i32, i32, i32, i32, i32, i32]),
        "tree_attention_paged": (i32, [vp, vp, vp, i32, vp, i32, i32, vp, vp, vp, tp, i32, i32, i32, i32, f32, i32,
                                       vp, vp, vp, sz, vp]),
        "tree_accept_workspace_size": (sz, [i32, tp, i32, i32]),
        "tree_accept": (i32, [i32, vp, vp, vp, tp, i32, i32, f32, u64, u64, vp, vp, vp, vp, vp, sz, vp]),
        "tree_accept_typical": (i32, [vp, vp, tp, i32, i32, f32, f32, f32, u64, u64, vp, vp, vp, vp, vp, sz, vp]),
        "tree_kv_commit_workspace_size": (sz, []),
        "tree_kv_commit": (i32, [vp, vp, vp, vp, vp, vp, vp, tp, i32, i32, i32, i32, i32, vp, sz, vp]),
        "tree_kv_commit_paged": (i32, [vp, vp, vp, vp, i32, vp, i32, i32, vp, vp, vp, tp, i32, i32, i32, i32, vp, sz,
                                       vp]),
        "spec_philox_uniform": (i32, [u64, u64, i32, i32, vp, vp, vp]),
        "spec_last_error": (ctypes.c_char_p, []),
        "spec_read_device_status": (i32, [vp, _i32p, vp]),
        "spec_selftest_timeout": (i32, [vp, u64, vp]),
        "spec_trace_begin": (i32, [i32]),
        "spec_trace_end": (i32, [ctypes.POINTER(spec_trace_entry), i32]),
        "spec_launch_count": (ctypes.c_int64, []),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


_lib = _load()


def exported_names():
    return [n for n in dir(_lib) if not n.startswith("_")]


def _check(fn, status):
    if status != 0:
        raise SpecError(fn, status, _lib.spec_last_error().decode())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _dtype_code(t):
    if t.dtype == torch.float32:
        return SPEC_F32
    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    raise TypeError(f"float tensors must be float32 or bfloat16, got {t.dtype}")


def _need(t, name, dtype=None, ndim=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions, got {tuple(t.shape)}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    return t


def _workspace(nbytes, device, ws):
    if ws is not None:
        return ws   # its size is checked by the library (SPEC_EWORKSPACE)
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=device)


class Tree:
    """An encoded candidate tree: the C struct plus the device buffer it points into."""

    def __init__(self, struct, buf, parent, rank):
        self.struct = struct
        self.buf = buf
        self.parent = parent
        self.rank = rank

    @property
    def T(self):
        return self.struct.T

    @property
    def max_depth(self):
        return self.struct.max_depth

    def ref(self):
        return ctypes.byref(self.struct)


# ---------------------------------------------------------------- entry points

def spec_tree_device_bytes(T):
    return int(_lib.spec_tree_device_bytes(int(T)))


def spec_tree_build(parent, rank=None, device=None, stream=None):
    """Encode a parent-index tree (host sequences) into a Tree on `device`."""
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    par = (ctypes.c_int32 * len(parent))(*[int(x) for x in parent])
    rk = (ctypes.c_int32 * len(rank))(*[int(x) for x in rank]) if rank is not None else None
    T = len(parent)
    nbytes = max(spec_tree_device_bytes(T), 16)
    buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
    st = spec_tree()
    with torch.cuda.device(device):
        _check("spec_tree_build", _lib.spec_tree_build(par, rk, T, _ptr(buf), nbytes, ctypes.byref(st), _stream(stream)))
    return Tree(st, buf, list(parent), None if rank is None else list(rank))


def hydra_draft_workspace_size(tree, B, d, V, cond, topk, dtype):
    K = len(cond)
    c = (ctypes.c_int32 * K)(*[int(x) for x in cond])
    k = (ctypes.c_int32 * K)(*[int(x) for x in topk])
    n = _lib.hydra_draft_workspace_size(tree.ref(), B, d, V, K, c, k, dtype)
    if n == 0:
        raise SpecError("hydra_draft_workspace_size", 1, _lib.spec_last_error().decode())
    return int(n)


def hydra_fold_embedding(W1, emb, out=None, stream=None):
    """The folded embedding table of a cond-1 head: fp32 [V, d], tab[v] = W1[:, d:] @ emb[v]."""
    _need(emb, "emb", ndim=2)
    dev = emb.device
    V, d = emb.shape
    _need(W1, "W1", dtype=emb.dtype, ndim=2, device=dev)
    if tuple(W1.shape) != (d, 2 * d):
        raise ValueError("W1 must be [d, 2d]")
    if _lib.hydra_fold_table_bytes(d, V) == 0:
        raise SpecError("hydra_fold_table_bytes", 1, _lib.spec_last_error().decode())
    if out is None:
        out = torch.empty(V, d, dtype=torch.float32, device=dev)
    _need(out, "out", dtype=torch.float32, ndim=2, device=dev)
    if tuple(out.shape) != (V, d):
        raise ValueError("out must be [V, d]")
    with torch.cuda.device(dev):
        _check("hydra_fold_embedding", _lib.hydra_fold_embedding(_ptr(W1), _ptr(emb), d, V, _dtype_code(emb), _ptr(out),
                                                                 _stream(stream)))
    return out


def hydra_draft(h, emb, W1, b1, W2, cond, topk, root_tok, tree, node_tok=None, node_logit=None,
                node_logprob=None, want_logprob=True, ws=None, stream=None, folded=None):
    """Fill the candidate tree: returns (node_tok [B,T] int32, node_logit [B,T], node_logprob [B,T] or None).

    folded: optional list (one entry per head, None allowed) of hydra_fold_embedding tables; cond-1
    heads with a table stream only the h_b half of W1 per call (hydra_draft_folded)."""
    _need(h, "h", ndim=2)
    dev = h.device
    dt = _dtype_code(h)
    B, d = h.shape
    _need(emb, "emb", dtype=h.dtype, ndim=2, device=dev)
    V = emb.shape[0]
    if emb.shape[1] != d:
        raise ValueError("emb must be [V, d]")
    K = len(W1)
    if len(W2) != K or len(cond) != K or len(topk) != K or (b1 is not None and len(b1) != K):
        raise ValueError("W1, b1, W2, cond and topk need one entry per head")
    for k in range(K):
        _need(W1[k], f"W1[{k}]", dtype=h.dtype, ndim=2, device=dev)
        d_in = d * (2 if cond[k] == 1 else (k + 1) if cond[k] == 2 else 1)
        if tuple(W1[k].shape) != (d, d_in):
            raise ValueError(f"W1[{k}] must be [d, {d_in // d}d] for cond {cond[k]}")
        _need(W2[k], f"W2[{k}]", dtype=h.dtype, ndim=2, device=dev)
        if tuple(W2[k].shape) != (V, d):
            raise ValueError(f"W2[{k}] must be [V, d]")
        if b1 is not None and b1[k] is not None:
            _need(b1[k], f"b1[{k}]", dtype=h.dtype, ndim=1, device=dev)
            if b1[k].shape[0] != d:
                raise ValueError(f"b1[{k}] must be [d]")
    _need(root_tok, "root_tok", dtype=torch.int32, ndim=1, device=dev)
    T = tree.T
    if node_tok is None:
        node_tok = torch.empty(B, T, dtype=torch.int32, device=dev)
    if node_logit is None:
        node_logit = torch.empty(B, T, dtype=torch.float32, device=dev)
    if node_logprob is None and want_logprob:
        node_logprob = torch.empty(B, T, dtype=torch.float32, device=dev)
    w1p = (ctypes.c_void_p * K)(*[W1[k].data_ptr() for k in range(K)])
    w2p = (ctypes.c_void_p * K)(*[W2[k].data_ptr() for k in range(K)])
    b1p = None if b1 is None else (ctypes.c_void_p * K)(*[(b1[k].data_ptr() if b1[k] is not None else 0) for k in range(K)])
    c = (ctypes.c_int32 * K)(*[int(x) for x in cond])
    kk = (ctypes.c_int32 * K)(*[int(x) for x in topk])
    nws = _lib.hydra_draft_workspace_size(tree.ref(), B, d, V, K, c, kk, dt)
    if nws == 0:
        raise SpecError("hydra_draft_workspace_size", 1, _lib.spec_last_error().decode())
    ws = _workspace(nws, dev, ws)
    if folded is not None:
        if len(folded) != K:
            raise ValueError("folded needs one entry per head")
        for k in range(K):
            if folded[k] is not None:
                _need(folded[k], f"folded[{k}]", dtype=torch.float32, ndim=2, device=dev)
                if tuple(folded[k].shape) != (V, d):
                    raise ValueError(f"folded[{k}] must be [V, d]")
        tabp = (ctypes.c_void_p * K)(*[(folded[k].data_ptr() if folded[k] is not None else 0) for k in range(K)])
        with torch.cuda.device(dev):
            _check("hydra_draft_folded", _lib.hydra_draft_folded(
                _ptr(h), _ptr(emb), K, w1p, b1p, w2p, tabp, c, kk, _ptr(root_tok), tree.ref(), B, d, V, dt,
                _ptr(node_tok), _ptr(node_logit), _ptr(node_logprob), _ptr(ws), ws.numel(), _stream(stream)))
        return node_tok, node_logit, node_logprob
    with torch.cuda.device(dev):
        _check("hydra_draft", _lib.hydra_draft(_ptr(h), _ptr(emb), K, w1p, b1p, w2p, c, kk, _ptr(root_tok), tree.ref(),
                                               B, d, V, dt, _ptr(node_tok), _ptr(node_logit), _ptr(node_logprob),
                                               _ptr(ws), ws.numel(), _stream(stream)))
    return node_tok, node_logit, node_logprob


def hydra_draft_folded(h, emb, W1, b1, W2, tab, cond, topk, root_tok, tree, **kw):
    """hydra_draft with the folded tables tab (one per head, None allowed) from hydra_fold_embedding."""
    return hydra_draft(h, emb, W1, b1, W2, cond, topk, root_tok, tree, folded=tab, **kw)


def hydra_draft_heads(h, emb, heads, root_tok, tree, ln_eps=1e-5, node_tok=None, node_logit=None, node_logprob=None,
                      want_logprob=True, ws=None, stream=None):
    """hydra_draft with one dict per head: cond, topk, form (0/1), W1, W2 and optionally b1, W1b, b1b, gamma, beta.

    Returns (node_tok, node_logit, node_logprob)."""
    _need(h, "h", ndim=2)
    dev = h.device
    dt = _dtype_code(h)
    B, d = h.shape
    _need(emb, "emb", dtype=h.dtype, ndim=2, device=dev)
    V = emb.shape[0]
    if emb.shape[1] != d:
        raise ValueError("emb must be [V, d]")
    K = len(heads)
    arr = (spec_head * K)()
    for k, hd in enumerate(heads):
        W1 = hd["W1"]
        _need(W1, f"heads[{k}].W1", dtype=h.dtype, ndim=2, device=dev)
        hidden = W1.shape[0]
        cond = int(hd["cond"])
        d_in = d * (2 if cond == 1 else (k + 1) if cond == 2 else 1)
        if W1.shape[1] != d_in:
            raise ValueError(f"heads[{k}].W1 must have {d_in} columns for cond {cond}")
        shapes = {"W2": (V, d), "b1": (hidden,), "W1b": (d, hidden), "b1b": (d,), "gamma": (d,), "beta": (d,)}
        for name, shp in shapes.items():
            t = hd.get(name)
            if t is not None:
                _need(t, f"heads[{k}].{name}", dtype=h.dtype, ndim=len(shp), device=dev)
                if tuple(t.shape) != shp:
                    raise ValueError(f"heads[{k}].{name} must be {shp}")
        arr[k].cond, arr[k].topk, arr[k].form, arr[k].hidden = cond, int(hd["topk"]), int(hd.get("form", 0)), hidden
        for name in ("W1", "b1", "W1b", "b1b", "gamma", "beta", "W2"):
            t = hd.get(name)
            setattr(arr[k], name, t.data_ptr() if t is not None else None)
    _need(root_tok, "root_tok", dtype=torch.int32, ndim=1, device=dev)
    T = tree.T
    if node_tok is None:
        node_tok = torch.empty(B, T, dtype=torch.int32, device=dev)
    if node_logit is None:
        node_logit = torch.empty(B, T, dtype=torch.float32, device=dev)
    if node_logprob is None and want_logprob:
        node_logprob = torch.empty(B, T, dtype=torch.float32, device=dev)
    nws = _lib.hydra_draft_heads_workspace_size(tree.ref(), B, d, V, K, arr, dt)
    if nws == 0:
        raise SpecError("hydra_draft_heads_workspace_size", 1, _lib.spec_last_error().decode())
    ws = _workspace(nws, dev, ws)
    with torch.cuda.device(dev):
        _check("hydra_draft_heads", _lib.hydra_draft_heads(_ptr(h), _ptr(emb), K, arr, _ptr(root_tok), tree.ref(), B, d,
                                                           V, float(ln_eps), dt, _ptr(node_tok), _ptr(node_logit),
                                                           _ptr(node_logprob), _ptr(ws), ws.numel(), _stream(stream)))
    return node_tok, node_logit, node_logprob


def tree_attention_workspace_size(tree, B, Hq, Hkv, Lmax, D, dtype):
    n = _lib.tree_attention_workspace_size(tree.ref(), B, Hq, Hkv, Lmax, D, dtype)
    if n == 0:
        raise SpecError("tree_attention_workspace_size", 1, _lib.spec_last_error().decode())
    return int(n)


def tree_attention(q, k_cache, v_cache, prefix_len, k_tree, v_tree, tree, scale=None, out=None, lse=None,
                   want_lse=True, ws=None, stream=None):
    """Tree attention: returns (out [B,Hq,T,D] float32, lse [B,Hq,T] float32 or None)."""
    _need(q, "q", ndim=4)
    dev = q.device
    dt = _dtype_code(q)
    B, Hq, T, D = q.shape
    _need(k_cache, "k_cache", dtype=q.dtype, ndim=4, device=dev)
    _need(v_cache, "v_cache", dtype=q.dtype, ndim=4, device=dev)
    Hkv, Lmax = k_cache.shape[1], k_cache.shape[2]
    if tuple(k_cache.shape) != (B, Hkv, Lmax, D) or tuple(v_cache.shape) != (B, Hkv, Lmax, D):
        raise ValueError("caches must be [B, Hkv, Lmax, D]")
    _need(k_tree, "k_tree", dtype=q.dtype, ndim=4, device=dev)
    _need(v_tree, "v_tree", dtype=q.dtype, ndim=4, device=dev)
    if tuple(k_tree.shape) != (B, Hkv, T, D) or tuple(v_tree.shape) != (B, Hkv, T, D):
        raise ValueError("tree keys/values must be [B, Hkv, T, D]")
    if T != tree.T:
        raise ValueError(f"q has {T} nodes, the tree {tree.T}")
    _need(prefix_len, "prefix_len", dtype=torch.int32, ndim=1, device=dev)
    if scale is None:
        scale = 0.0   # the library's default, 1/sqrt(D)
    if out is None:
        out = torch.empty(B, Hq, T, D, dtype=torch.float32, device=dev)
    if lse is None and want_lse:
        lse = torch.empty(B, Hq, T, dtype=torch.float32, device=dev)
    nws = _lib.tree_attention_workspace_size(tree.ref(), B, Hq, Hkv, Lmax, D, dt)
    if nws == 0:
        raise SpecError("tree_attention_workspace_size", 1, _lib.spec_last_error().decode())
    ws = _workspace(nws, dev, ws)
    with torch.cuda.device(dev):
        _check("tree_attention", _lib.tree_attention(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(prefix_len),
                                                     _ptr(k_tree), _ptr(v_tree), tree.ref(), B, Hq, Hkv, Lmax, D,
                                                     float(scale), dt, _ptr(out), _ptr(lse), _ptr(ws), ws.numel(),
                                                     _stream(stream)))
    return out, lse


def tree_attention_paged_workspace_size(tree, B, Hq, Hkv, max_blocks, block_size, D, dt):
    n = _lib.tree_attention_paged_workspace_size(tree.ref(), B, Hq, Hkv, max_blocks, block_size, D, dt)
    if n == 0:
        raise SpecError("tree_attention_paged_workspace_size", 1, _lib.spec_last_error().decode())
    return int(n)


def tree_attention_paged(q, k_pool, v_pool, block_table, prefix_len, k_tree, v_tree, tree, scale=None, out=None,
                         lse=None, want_lse=True, ws=None, stream=None):
    """Tree attention over a paged cache: pools [num_blocks, Hkv, block_size, D], block_table [B, max_blocks] int32."""
    _need(q, "q", ndim=4)
    dev = q.device
    dt = _dtype_code(q)
    B, Hq, T, D = q.shape
    _need(k_pool, "k_pool", dtype=q.dtype, ndim=4, device=dev)
    _need(v_pool, "v_pool", dtype=q.dtype, ndim=4, device=dev)
    num_blocks, Hkv, bs = k_pool.shape[0], k_pool.shape[1], k_pool.shape[2]
    if tuple(k_pool.shape) != (num_blocks, Hkv, bs, D) or tuple(v_pool.shape) != (num_blocks, Hkv, bs, D):
        raise ValueError("pools must be [num_blocks, Hkv, block_size, D]")
    _need(block_table, "block_table", dtype=torch.int32, ndim=2, device=dev)
    if block_table.shape[0] != B:
        raise ValueError("block_table must be [B, max_blocks]")
    max_blocks = block_table.shape[1]
    _need(k_tree, "k_tree", dtype=q.dtype, ndim=4, device=dev)
    _need(v_tree, "v_tree", dtype=q.dtype, ndim=4, device=dev)
    if tuple(k_tree.shape) != (B, Hkv, T, D) or tuple(v_tree.shape) != (B, Hkv, T, D):
        raise ValueError("tree keys/values must be [B, Hkv, T, D]")
    if T != tree.T:
        raise ValueError(f"q has {T} nodes, the tree {tree.T}")
    _need(prefix_len, "prefix_len", dtype=torch.int32, ndim=1, device=dev)
    if scale is None:
        scale = 0.0   # the library's default, 1/sqrt(D)
    if out is None:
        out = torch.empty(B, Hq, T, D, dtype=torch.float32, device=dev)
    if lse is None and want_lse:
        lse = torch.empty(B, Hq, T, dtype=torch.float32, device=dev)
    nws = _lib.tree_attention_paged_workspace_size(tree.ref(), B, Hq, Hkv, max_blocks, bs, D, dt)
    if nws == 0:
        raise SpecError("tree_attention_paged_workspace_size", 1, _lib.spec_last_error().decode())
    ws = _workspace(nws, dev, ws)
    with torch.cuda.device(dev):
        _check("tree_attention_paged", _lib.tree_attention_paged(
            _ptr(q), _ptr(k_pool), _ptr(v_pool), num_blocks, _ptr(block_table), max_blocks, bs, _ptr(prefix_len),
            _ptr(k_tree), _ptr(v_tree), tree.ref(), B, Hq, Hkv, D, float(scale), dt, _ptr(out), _ptr(lse), _ptr(ws),
            ws.numel(), _stream(stream)))
    return out, lse


def tree_attention_noalloc(q, k_cache, v_cache, prefix_len, k_tree, v_tree, tree, scale=None, out=None, lse=None,
                           want_lse=True, stream=None):
    """tree_attention for callers that cannot allocate device scratch: the library's
    built-in 32 MiB buffer serves as workspace (one call at a time per process).
    Outputs are allocated here only when the caller passes none."""
    _need(q, "q", ndim=4)
    dev = q.device
    dt = _dtype_code(q)
    B, Hq, T, D = q.shape
    _need(k_cache, "k_cache", dtype=q.dtype, ndim=4, device=dev)
    _need(v_cache, "v_cache", dtype=q.dtype, ndim=4, device=dev)
    Hkv, Lmax = k_cache.shape[1], k_cache.shape[2]
    if tuple(k_cache.shape) != (B, Hkv, Lmax, D) or tuple(v_cache.shape) != (B, Hkv, Lmax, D):
        raise ValueError("caches must be [B, Hkv, Lmax, D]")
    _need(k_tree, "k_tree", dtype=q.dtype, ndim=4, device=dev)
    _need(v_tree, "v_tree", dtype=q.dtype, ndim=4, device=dev)
    if tuple(k_tree.shape) != (B, Hkv, T, D) or tuple(v_tree.shape) != (B, Hkv, T, D):
        raise ValueError("tree keys/values must be [B, Hkv, T, D]")
    if T != tree.T:
        raise ValueError(f"q has {T} nodes, the tree {tree.T}")
    _need(prefix_len, "prefix_len", dtype=torch.int32, ndim=1, device=dev)
    if scale is None:
        scale = 0.0   # the library's default, 1/sqrt(D)
    if out is None:
        out = torch.empty(B, Hq, T, D, dtype=torch.float32, device=dev)
    if lse is None and want_lse:
        lse = torch.empty(B, Hq, T, dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        _check("tree_attention_noalloc", _lib.tree_attention_noalloc(
            _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(prefix_len), _ptr(k_tree), _ptr(v_tree), tree.ref(),
            B, Hq, Hkv, Lmax, D, float(scale), dt, _ptr(out), _ptr(lse), _stream(stream)))
    return out, lse


def tree_attention_noalloc_status(device=None, stream=None):
    """Status word of the built-in scratch tree_attention_noalloc uses (0 = no failure)."""
    v = ctypes.c_int32(0)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        _check("tree_attention_noalloc_status", _lib.tree_attention_noalloc_status(ctypes.byref(v), _stream(stream)))
    return v.value


def tree_accept_workspace_size(mode, tree, B, V):
    n = _lib.tree_accept_workspace_size(int(mode), tree.ref(), B, V)
    if n == 0:
        raise SpecError("tree_accept_workspace_size", 1, _lib.spec_last_error().decode())
    return int(n)


def tree_accept(mode, logits_p, logits_q, node_tok, tree, temperature=1.0, seed=0, offset=0, accept_len=None,
                accept_path=None, next_token=None, margin=None, want_margin=True, ws=None, stream=None):
    """Acceptance (mode 0 greedy, 1 rejection): returns (accept_len, accept_path, next_token, margin)."""
    _need(logits_p, "logits_p", dtype=torch.float32, ndim=3)
    dev = logits_p.device
    B, T, V = logits_p.shape
    if T != tree.T:
        raise ValueError(f"logits have {T} nodes, the tree {tree.T}")
    if mode == 1:
        _need(logits_q, "logits_q", dtype=torch.float32, ndim=3, device=dev)
        if tuple(logits_q.shape) != (B, T, V):
            raise ValueError("logits_q must match logits_p")
    _need(node_tok, "node_tok", dtype=torch.int32, ndim=2, device=dev)
    if tuple(node_tok.shape) != (B, T):
        raise ValueError("node_tok must be [B, T]")
    if accept_len is None:
        accept_len = torch.empty(B, dtype=torch.int32, device=dev)
    if accept_path is None:
        accept_path = torch.empty(B, tree.max_depth + 1, dtype=torch.int32, device=dev)
    if next_token is None:
        next_token = torch.empty(B, dtype=torch.int32, device=dev)
    if margin is None and want_margin:
        margin = torch.empty(B, dtype=torch.float32, device=dev)
    nws = _lib.tree_accept_workspace_size(int(mode), tree.ref(), B, V)
    if nws == 0:
        raise SpecError("tree_accept_workspace_size", 1, _lib.spec_last_error().decode())
    ws = _workspace(nws, dev, ws)
    with torch.cuda.device(dev):
        _check("tree_accept", _lib.tree_accept(int(mode), _ptr(logits_p), _ptr(logits_q if mode == 1 else None),
                                               _ptr(node_tok), tree.ref(), B, V, float(temperature), int(seed),
                                               int(offset), _ptr(accept_len), _ptr(accept_path), _ptr(next_token),
                                               _ptr(margin), _ptr(ws), ws.numel(), _stream(stream)))
    return accept_len, accept_path, next_token, margin


def tree_kv_commit_workspace_size():
    return int(_lib.tree_kv_commit_workspace_size())


def tree_kv_commit(k_tree, v_tree, k_cache, v_cache, prefix_len, accept_len, accept_path, tree, ws=None,
                   stream=None):
    """Append the accepted path's K/V rows to the caches and advance prefix_len, in place."""
    _need(k_tree, "k_tree", ndim=4)
    dev = k_tree.device
    B, Hkv, T, D = k_tree.shape
    if T != tree.T:
        raise ValueError(f"k_tree has {T} nodes, the tree {tree.T}")
    for name, t in (("v_tree", v_tree), ("k_cache", k_cache), ("v_cache", v_cache)):
        _need(t, name, dtype=k_tree.dtype, ndim=4, device=dev)
    if tuple(v_tree.shape) != (B, Hkv, T, D):
        raise ValueError("v_tree must match k_tree")
    Lmax = k_cache.shape[2]
    if tuple(k_cache.shape) != (B, Hkv, Lmax, D) or tuple(v_cache.shape) != (B, Hkv, Lmax, D):
        raise ValueError("caches must be [B, Hkv, Lmax, D] with the tree's B, Hkv and D")
    _need(prefix_len, "prefix_len", dtype=torch.int32, ndim=1, device=dev)
    _need(accept_len, "accept_len", dtype=torch.int32, ndim=1, device=dev)
    _need(accept_path, "accept_path", dtype=torch.int32, ndim=2, device=dev)
    if prefix_len.shape[0] != B or accept_len.shape[0] != B or tuple(accept_path.shape) != (B, tree.max_depth + 1):
        raise ValueError("prefix_len, accept_len [B] and accept_path [B, max_depth + 1] must match")
    dt = _dtype_code(k_tree)
    ws = _workspace(int(_lib.tree_kv_commit_workspace_size()), dev, ws)
    with torch.cuda.device(dev):
        _check("tree_kv_commit", _lib.tree_kv_commit(_ptr(k_tree), _ptr(v_tree), _ptr(k_cache), _ptr(v_cache),
                                                     _ptr(prefix_len), _ptr(accept_len), _ptr(accept_path),
                                                     tree.ref(), B, Hkv, Lmax, D, dt, _ptr(ws), ws.numel(),
                                                     _stream(stream)))
    return ws


def tree_kv_commit_paged(k_tree, v_tree, k_pool, v_pool, block_table, block_size, prefix_len, accept_len,
                         accept_path, tree, ws=None, stream=None):
    """tree_kv_commit into a paged cache: pool [num_blocks, Hkv, block_size, D], block_table [B, max_blocks]."""
    _need(k_tree, "k_tree", ndim=4)
    dev = k_tree.device
    B, Hkv, T, D = k_tree.shape
    if T != tree.T:
        raise ValueError(f"k_tree has {T} nodes, the tree {tree.T}")
    for name, t in (("v_tree", v_tree), ("k_pool", k_pool), ("v_pool", v_pool)):
        _need(t, name, dtype=k_tree.dtype, ndim=4, device=dev)
    if tuple(v_tree.shape) != (B, Hkv, T, D):
        raise ValueError("v_tree must match k_tree")
    num_blocks = k_pool.shape[0]
    if tuple(k_pool.shape) != (num_blocks, Hkv, block_size, D) or tuple(v_pool.shape) != tuple(k_pool.shape):
        raise ValueError("pools must be [num_blocks, Hkv, block_size, D] with the tree's Hkv and D")
    _need(block_table, "block_table", dtype=torch.int32, ndim=2, device=dev)
    if block_table.shape[0] != B:
        raise ValueError("block_table must be [B, max_blocks]")
    _need(prefix_len, "prefix_len", dtype=torch.int32, ndim=1, device=dev)
    _need(accept_len, "accept_len", dtype=torch.int32, ndim=1, device=dev)
    _need(accept_path, "accept_path", dtype=torch.int32, ndim=2, device=dev)
    if prefix_len.shape[0] != B or accept_len.shape[0] != B or tuple(accept_path.shape) != (B, tree.max_depth + 1):
        raise ValueError("prefix_len, accept_len [B] and accept_path [B, max_depth + 1] must match")
    dt = _dtype_code(k_tree)
    ws = _workspace(int(_lib.tree_kv_commit_workspace_size()), dev, ws)
    with torch.cuda.device(dev):
        _check("tree_kv_commit_paged", _lib.tree_kv_commit_paged(
            _ptr(k_tree), _ptr(v_tree), _ptr(k_pool), _ptr(v_pool), num_blocks, _ptr(block_table),
            block_table.shape[1], block_size, _ptr(prefix_len), _ptr(accept_len), _ptr(accept_path), tree.ref(), B, Hkv,
            D, dt, _ptr(ws), ws.numel(), _stream(stream)))
    return ws


def tree_accept_typical(logits_p, node_tok, tree, temperature=1.0, epsilon=0.09, alpha=0.3, seed=0, offset=0,
                        accept_len=None, accept_path=None, next_token=None, margin=None, want_margin=True, ws=None,
                        stream=None):
    """Typical acceptance: returns (accept_len, accept_path, next_token, margin)."""
    _need(logits_p, "logits_p", dtype=torch.float32, ndim=3)
    dev = logits_p.device
    B, T, V = logits_p.shape
    if T != tree.T:
        raise ValueError(f"logits have {T} nodes, the tree {tree.T}")
    _need(node_tok, "node_tok", dtype=torch.int32, ndim=2, device=dev)
    if tuple(node_tok.shape) != (B, T):
        raise ValueError("node_tok must be [B, T]")
    if accept_len is None:
        accept_len = torch.empty(B, dtype=torch.int32, device=dev)
    if accept_path is None:
        accept_path = torch.empty(B, tree.max_depth + 1, dtype=torch.int32, device=dev)
    if next_token is None:
        next_token = torch.empty(B, dtype=torch.int32, device=dev)
    if margin is None and want_margin:
        margin = torch.empty(B, dtype=torch.float32, device=dev)
    nws = _lib.tree_accept_workspace_size(2, tree.ref(), B, V)
    if nws == 0:
        raise SpecError("tree_accept_workspace_size", 1, _lib.spec_last_error().decode())
    ws = _workspace(nws, dev, ws)
    with torch.cuda.device(dev):
        _check("tree_accept_typical", _lib.tree_accept_typical(
            _ptr(logits_p), _ptr(node_tok), tree.ref(), B, V, float(temperature), float(epsilon), float(alpha),
            int(seed), int(offset), _ptr(accept_len), _ptr(accept_path), _ptr(next_token), _ptr(margin), _ptr(ws),
            ws.numel(), _stream(stream)))
    return accept_len, accept_path, next_token, margin


def spec_philox_uniform(seed, offset, B, T, device=None, stream=None):
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    ua = torch.empty(B, T, dtype=torch.float32, device=device)
    us = torch.empty(B, dtype=torch.float32, device=device)
    with torch.cuda.device(device):
        _check("spec_philox_uniform", _lib.spec_philox_uniform(int(seed), int(offset), B, T, _ptr(ua), _ptr(us),
                                                               _stream(stream)))
    return ua, us


def spec_read_device_status(ws, stream=None):
    v = ctypes.c_int32(0)
    _check("spec_read_device_status", _lib.spec_read_device_status(_ptr(ws), ctypes.byref(v), _stream(stream)))
    return v.value


def spec_selftest_timeout(ws, limit_ns=1_000_000, stream=None):
    """Run the bounded-wait self-test kernel on `ws` (a CUDA uint8 tensor >= 16 bytes)."""
    _need(ws, "ws")
    with torch.cuda.device(ws.device):
        _check("spec_selftest_timeout", _lib.spec_selftest_timeout(_ptr(ws), int(limit_ns), _stream(stream)))


def spec_last_error():
    return _lib.spec_last_error().decode()


def spec_trace_begin(capacity=4096):
    _check("spec_trace_begin", _lib.spec_trace_begin(int(capacity)))


def spec_trace_end(max_entries=64):
    arr = (spec_trace_entry * max_entries)()
    n = _lib.spec_trace_end(arr, max_entries)
    if n < 0:
        raise SpecError("spec_trace_end", 1, _lib.spec_last_error().decode())
    return {arr[i].name.decode(): (arr[i].launches, arr[i].total_ms) for i in range(min(n, max_entries))}


def spec_launch_count():
    return int(_lib.spec_launch_count())
