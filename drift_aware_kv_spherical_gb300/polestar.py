"""Thin Python binding of libpolestar's C ABI (include/polestar.h).

Argument marshalling only: every function below forwards torch device
tensors as raw pointers to the function of the same name in libpolestar.so,
and every step of the computation runs in its CUDA kernels.  There is no CPU
path: if the library is missing or a call fails, a PolestarError is raised.
"""

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpolestar.so")

PS_OK, PS_ERR_ARG, PS_ERR_UNSUPPORTED, PS_ERR_WORKSPACE, PS_ERR_CUDA, PS_ERR_TIMEOUT = range(6)
PS_F32, PS_BF16 = 0, 1
OP_KMEANS, OP_NVFP4, OP_PROXY_KL, OP_TOPK, OP_REFRESH, OP_COMMIT = range(6)
EXPORTED = ["ps_create", "ps_destroy", "ps_check", "ps_status_string", "ps_last_cuda_error",
            "ps_trace_enable", "ps_trace_count", "ps_trace_get",
            "ps_workspace_bytes", "ps_kmeans_spherical", "ps_nvfp4_residual",
            "ps_proxy_attn_kl", "ps_topk_drift", "ps_refresh_kv", "ps_commit",
            "ps_store_record_bytes", "ps_host_alloc", "ps_host_free",
            "ps_nvfp4_pack_clusters", "ps_nvfp4_fetch_dequant", "ps_schedule_step", "ps_drift_score",
            "ps_block_progress"]

_p = ctypes.c_void_p
_i = ctypes.c_int
_sz = ctypes.c_size_t


class PolestarError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        lib = Library.load()
        msg = f"{where}: {lib.status_string(status)} ({status})"
        if status == PS_ERR_CUDA:
            msg += f" [{lib.cdll.ps_last_cuda_error().decode()}]"
        super().__init__(msg)


class CommitParams(ctypes.Structure):
    _fields_ = [("tau_s", ctypes.c_float), ("alpha", ctypes.c_float),
                ("ratio", ctypes.c_float), ("mode", ctypes.c_int),
                ("ensure_progress", ctypes.c_int)]


class ScheduleParams(ctypes.Structure):
    _fields_ = [("tau_upd", ctypes.c_int), ("full_period", ctypes.c_int),
                ("block_len", ctypes.c_int)]


class ScheduleState(ctypes.Structure):
    _fields_ = [("since", ctypes.c_int), ("refreshes", ctypes.c_int),
                ("block_start", ctypes.c_int)]


SCHED_REFRESH, SCHED_FULL, SCHED_SLIDE, SCHED_REINIT = 1, 2, 4, 8
SCORER_KL, SCORER_COSINE, SCORER_ENTROPY = 0, 1, 2

_SIGS = {
    "ps_create": (_i, [_i, ctypes.POINTER(_p)]),
    "ps_destroy": (_i, [_p]),
    "ps_check": (_i, [_p, _p, _i]),
    "ps_status_string": (ctypes.c_char_p, [_i]),
    "ps_last_cuda_error": (ctypes.c_char_p, []),
    "ps_trace_enable": (_i, [_p, _i]),
    "ps_trace_count": (_i, [_p]),
    "ps_trace_get": (_i, [_p, _i, ctypes.POINTER(ctypes.c_char_p),
                          ctypes.POINTER(ctypes.c_float)]),
    "ps_workspace_bytes": (_sz, [_i] * 11),
    "ps_store_record_bytes": (_sz, [_i]),
    "ps_host_alloc": (_i, [_sz, ctypes.POINTER(_p)]),
    "ps_host_free": (_i, [_p]),
    "ps_drift_score": (_i, [_p, _p, _p, _i, _i, _i, _i, _p, _p]),
    "ps_block_progress": (_i, [_p, _p, _p, _p, _i, _i, _p, _p]),
    "ps_schedule_step": (_i, [ctypes.POINTER(ScheduleParams), ctypes.POINTER(ScheduleState),
                              _i, _i]),
    "ps_nvfp4_pack_clusters": (_i, [_p, _p, _p, _p, _i, _i, _i, _i, _p, _p, _p, _p]),
    "ps_nvfp4_fetch_dequant": (_i, [_p, _p, _p, _p, _p, _i, _p, _p, _p, _i, _i, _i, _i, _p,
                                    _p]),
    "ps_kmeans_spherical": (_i, [_p, _p, _i, _i, _i, _i, _i, _i, _i, _p, _p, _p,
                                 _p, _p, _p, _p, _p, _sz, _p]),
    "ps_nvfp4_residual": (_i, [_p, _p, _i, _p, _p, _p, _i, _i, _i, _i, _p, _p, _p,
                               _p, _sz, _p]),
    "ps_proxy_attn_kl": (_i, [_p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i, _p,
                              _p, _p, _p, _sz, _p]),
    "ps_topk_drift": (_i, [_p, _p, _p, _p, _i, _i, _i, _i, _p, _p, _p, _p, _p, _p,
                           _sz, _p]),
    "ps_refresh_kv": (_i, [_p, _p, _i, _p, _p, _p, _p, _i, _i, _i, _i, _i, _p, _p,
                           _i, _i, _p, _sz, _p]),
    "ps_commit": (_i, [_p, _p, _i, _i, _i, _i, _p, _p, _p, _i, _p, _p, _p, _p, _i,
                       CommitParams, _p, _p, _p, _p, _sz, _p]),
}


class Library:
    """The loaded libpolestar.so (one per process)."""

    _inst = None

    def __init__(self, path):
        self.cdll = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(self.cdll, name)
            fn.restype = res
            fn.argtypes = args
        self.path = path
        self._handles = {}

    @classmethod
    def load(cls, path=None):
        if cls._inst is None:
            path = path or LIB_PATH
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is not built; run `python -c 'import __graft_entry__ as g; "
                    "g.build()'` (libpolestar has no CPU fallback)")
            cls._inst = cls(path)
        return cls._inst

    def status_string(self, s):
        return self.cdll.ps_status_string(s).decode()

    def handle(self, device=None):
        """A process-wide handle for `device` (created on first use)."""
        dev = torch.cuda.current_device() if device is None else int(device)
        if dev not in self._handles:
            h = _p()
            st = self.cdll.ps_create(dev, ctypes.byref(h))
            if st != PS_OK:
                raise PolestarError(st, "ps_create")
            self._handles[dev] = h
        return self._handles[dev]


def _lib():
    return Library.load()


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libpolestar takes device tensors only")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def _dtype(t):
    if t.dtype == torch.float32:
        return PS_F32
    if t.dtype == torch.bfloat16:
        return PS_BF16
    raise ValueError(f"unsupported dtype {t.dtype}")


def _check(st, where):
    if st != PS_OK:
        raise PolestarError(st, where)


def _ws(ws):
    return (None, 0) if ws is None else (ws.data_ptr(), ws.numel() * ws.element_size())


def ps_workspace_bytes(op, B=0, N=0, d=0, C=0, Hq=0, Hkv=0, dh=0, k=0, P=0, V=0):
    return int(_lib().cdll.ps_workspace_bytes(op, B, N, d, C, Hq, Hkv, dh, k, P, V))


def workspace(op, device=None, **sizes):
    """A caller-owned workspace tensor large enough for `op` at `sizes`."""
    n = ps_workspace_bytes(op, **sizes)
    if n == 0:
        return None
    return torch.empty(n, dtype=torch.uint8,
                       device=device if device is not None else "cuda")


def ps_check(synchronize=True, stream=None):
    lib = _lib()
    _check(lib.cdll.ps_check(lib.handle(), _stream(stream), int(synchronize)), "ps_check")


def ps_kmeans_spherical(H, mu, assign, rho, chat, counts, iters, init_mode=0,
                        init_u=None, objective=None, ws=None, stream=None):
    lib = _lib()
    B, N, d = H.shape
    C = mu.shape[1]
    w, wn = _ws(ws)
    st = lib.cdll.ps_kmeans_spherical(
        lib.handle(), _ptr(H), _dtype(H), B, N, d, C, iters, init_mode,
        _ptr(init_u), _ptr(mu), _ptr(assign), _ptr(rho), _ptr(chat), _ptr(counts),
        _ptr(objective), w, wn, _stream(stream))
    _check(st, "ps_kmeans_spherical")


def ps_nvfp4_residual(H, mu, assign, rho, codes, scales, tensor_scale, ws=None,
                      stream=None):
    lib = _lib()
    B, N, d = H.shape
    C = mu.shape[1] if mu is not None else 1
    w, wn = _ws(ws)
    st = lib.cdll.ps_nvfp4_residual(
        lib.handle(), _ptr(H), _dtype(H), _ptr(mu), _ptr(assign), _ptr(rho), B, N,
        d, C, _ptr(codes), _ptr(scales), _ptr(tensor_scale), w, wn, _stream(stream))
    _check(st, "ps_nvfp4_residual")


def ps_proxy_attn_kl(Q, chat, Wk, A_prev, A_cur, D, Hkv, ws=None, stream=None):
    lib = _lib()
    B, N, Hq, dh = Q.shape
    C, d = chat.shape[1], chat.shape[2]
    w, wn = _ws(ws)
    st = lib.cdll.ps_proxy_attn_kl(
        lib.handle(), _ptr(Q), _ptr(chat), _ptr(Wk), _dtype(Q), B, N, d, C, Hq, Hkv,
        dh, _ptr(A_prev), _ptr(A_cur), _ptr(D), w, wn, _stream(stream))
    _check(st, "ps_proxy_attn_kl")


def ps_topk_drift(D, assign, counts, k, sel, sel_score, pos, npos, posmask=None,
                  ws=None, stream=None):
    lib = _lib()
    B, N = D.shape
    C = counts.shape[1]
    w, wn = _ws(ws)
    st = lib.cdll.ps_topk_drift(
        lib.handle(), _ptr(D), _ptr(assign), _ptr(counts), B, N, C, k, _ptr(sel),
        _ptr(sel_score), _ptr(pos), _ptr(npos), _ptr(posmask), w, wn, _stream(stream))
    _check(st, "ps_topk_drift")


def ps_refresh_kv(H, pos, npos, Wk, Wv, Kcache, Vcache, Hkv, dh, cache_off=0,
                  ws=None, stream=None):
    lib = _lib()
    B, N, d = H.shape
    Ncache = Kcache.shape[1]
    w, wn = _ws(ws)
    st = lib.cdll.ps_refresh_kv(
        lib.handle(), _ptr(H), _dtype(H), _ptr(pos), _ptr(npos), _ptr(Wk), _ptr(Wv),
        B, N, d, Hkv, dh, _ptr(Kcache), _ptr(Vcache), Ncache, cache_off, w, wn,
        _stream(stream))
    _check(st, "ps_refresh_kv")


def ps_commit(logits, role, undecided, D_blk, d_ld, d_sum, d_cnt, d_prev,
              suffix_sel, sel_ld, params, token, conf, commit, ws=None,
              stream=None):
    lib = _lib()
    B, P, V = logits.shape
    w, wn = _ws(ws)
    if not isinstance(params, CommitParams):
        params = CommitParams(*params)
    st = lib.cdll.ps_commit(
        lib.handle(), _ptr(logits), _dtype(logits), B, P, V, _ptr(role), _ptr(undecided), _ptr(D_blk),
        d_ld, _ptr(d_sum), _ptr(d_cnt), _ptr(d_prev), _ptr(suffix_sel), sel_ld, params,
        _ptr(token), _ptr(conf), _ptr(commit), w, wn, _stream(stream))
    _check(st, "ps_commit")


def ps_drift_score(A_cur, A_prev, scorer, D, stream=None):
    """Ablation drift signal (SCORER_*) of distributions A_cur [B][N][C]
    against A_prev (or None) into D [B][N]."""
    lib = _lib()
    B, N, C = A_cur.shape
    st = lib.cdll.ps_drift_score(lib.handle(), _ptr(A_cur), _ptr(A_prev), B, N, C, int(scorer),
                                 _ptr(D), _stream(stream))
    _check(st, "ps_drift_score")


def ps_nvfp4_residual_noalloc(H, mu, assign, rho, codes, scales, tensor_scale,
                              stream=None):
    """ps_nvfp4_residual without a workspace: for callers that cannot
    allocate device memory; the library's fixed device array holds the
    scratch (B <= 16384; overlapping calls on one device race)."""
    lib = _lib()
    fn = lib.cdll.ps_nvfp4_residual_noalloc
    fn.restype = _i
    fn.argtypes = [_p, _p, _i, _p, _p, _p, _i, _i, _i, _i, _p, _p, _p, _p]
    B, N, d = H.shape
    C = mu.shape[1] if mu is not None else 1
    st = fn(lib.handle(), _ptr(H), _dtype(H), _ptr(mu), _ptr(assign), _ptr(rho), B, N,
            d, C, _ptr(codes), _ptr(scales), _ptr(tensor_scale), _stream(stream))
    _check(st, "ps_nvfp4_residual_noalloc")


def ps_trace_enable(enable=True):
    """Start (clearing earlier records) or stop the library's kernel trace."""
    lib = _lib()
    _check(lib.cdll.ps_trace_enable(lib.handle(), int(bool(enable))), "ps_trace_enable")


def ps_trace_records():
    """[(kernel name, ms)] for every kernel launched since tracing was enabled,
    in launch order (waits for them to finish)."""
    lib = _lib()
    out = []
    for i in range(lib.cdll.ps_trace_count(lib.handle())):
        name = ctypes.c_char_p()
        ms = ctypes.c_float()
        _check(lib.cdll.ps_trace_get(lib.handle(), i, ctypes.byref(name), ctypes.byref(ms)),
               "ps_trace_get")
        out.append((name.value.decode(), ms.value))
    return out


# ---- offload of the quantised clusters (include/polestar.h)
def ps_store_record_bytes(d):
    return int(_lib().cdll.ps_store_record_bytes(int(d)))


class HostStore:
    """Pinned host memory mapped into the device (ps_host_alloc): `ptr` is
    valid on host and device; `view()` is a numpy byte view of it."""

    def __init__(self, nbytes):
        lib = _lib()
        p = ctypes.c_void_p()
        _check(lib.cdll.ps_host_alloc(int(nbytes), ctypes.byref(p)), "ps_host_alloc")
        self.ptr, self.nbytes = p.value, int(nbytes)

    def view(self):
        import numpy as np
        buf = (ctypes.c_uint8 * self.nbytes).from_address(self.ptr)
        return np.frombuffer(buf, dtype=np.uint8)

    def free(self):
        if self.ptr:
            _check(_lib().cdll.ps_host_free(ctypes.c_void_p(self.ptr)), "ps_host_free")
            self.ptr = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


def _store_ptr(store):
    return store.ptr if isinstance(store, HostStore) else _ptr(store)


def ps_nvfp4_pack_clusters(codes, scales, assign, C, store, order, cl_off, stream=None):
    """Cluster-grouped records of every window into `store` (a device uint8
    tensor or a HostStore), with order [B][N] and cl_off [B][C+1] (int32)."""
    lib = _lib()
    B, N, half = codes.shape
    st = lib.cdll.ps_nvfp4_pack_clusters(lib.handle(), _ptr(codes), _ptr(scales), _ptr(assign),
                                         B, N, 2 * half, int(C), _store_ptr(store), _ptr(order),
                                         _ptr(cl_off), _stream(stream))
    _check(st, "ps_nvfp4_pack_clusters")


def ps_nvfp4_fetch_dequant(store, order, cl_off, sel, mu, rho, tensor_scale, Ht, stream=None):
    """Reconstructed rows of the selected clusters, read from `store`, into
    Ht [B][N][d] (bf16); other rows untouched."""
    lib = _lib()
    B, N, d = Ht.shape
    C = mu.shape[1]
    st = lib.cdll.ps_nvfp4_fetch_dequant(lib.handle(), _store_ptr(store), _ptr(order),
                                         _ptr(cl_off), _ptr(sel), sel.shape[1], _ptr(mu),
                                         _ptr(rho), _ptr(tensor_scale), B, N, d, C, _ptr(Ht),
                                         _stream(stream))
    _check(st, "ps_nvfp4_fetch_dequant")


def ps_block_progress(commit, undecided, role, out, stream=None):
    """(tokens committed, block decided) of a decode step into `out`: a
    HostStore of >= 8 bytes (readable on the host once `stream` has reached
    it) or an int32 device tensor of 2 elements."""
    lib = _lib()
    B, P = commit.shape
    st = lib.cdll.ps_block_progress(lib.handle(), _ptr(commit), _ptr(undecided), _ptr(role),
                                    B, P, _store_ptr(out), _stream(stream))
    _check(st, "ps_block_progress")


# ---- refresh schedule of the decode loop (include/polestar.h; host only)
def ps_schedule_step(params, state, committed, block_done):
    """Actions (SCHED_* flags) of the next step; updates `state` in place."""
    act = _lib().cdll.ps_schedule_step(ctypes.byref(params), ctypes.byref(state),
                                       int(committed), int(bool(block_done)))
    if act < 0:
        raise PolestarError(-act, "ps_schedule_step")
    return act


class Schedule:
    """A decode loop's schedule: tau_upd tokens between refreshes, every
    full_period-th refresh in full, the window sliding by block_len."""

    def __init__(self, tau_upd, full_period, block_len):
        self.params = ScheduleParams(int(tau_upd), int(full_period), int(block_len))
        self.state = ScheduleState(0, 0, 0)

    def step(self, committed, block_done):
        return ps_schedule_step(self.params, self.state, committed, block_done)
