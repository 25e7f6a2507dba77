"""ctypes binding of libeagle's C ABI (include/eagle.h), with the same names.

Argument marshalling only: every computation happens in the library's CUDA
kernels.  Pointers cross the boundary as plain integers (device addresses);
structs mirror the header field by field.  Loading fails loudly if the
library has not been built.
"""
from __future__ import annotations

import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libeagle.so")

EAGLE_MAX_NODES = 256
EAGLE_MAX_CHILDREN = 16
EAGLE_MAX_LAYERS = 128
EAGLE_MAX_VOCAB = 32768

PHASE_ROOT, PHASE_FRONTIER, PHASE_FINAL = 0, 1, 2

STATUS = {0: "EAGLE_OK", 1: "EAGLE_ERR_INVALID_ARG", 2: "EAGLE_ERR_SHAPE", 3: "EAGLE_ERR_ALIGN",
          4: "EAGLE_ERR_CAPACITY", 5: "EAGLE_ERR_INVALID_TREE", 6: "EAGLE_ERR_NUMERIC",
          7: "EAGLE_ERR_TIMEOUT", 8: "EAGLE_ERR_UNSUPPORTED", 9: "EAGLE_ERR_CUDA"}
STATUS_CODE = {v: k for k, v in STATUS.items()}

KERNEL_ID = {"all": -1, "gemm_fc": 0, "gemm_qkv": 1, "gemm_o": 2, "gemm_gateup": 3, "gemm_down": 4,
             "gemm_lm": 5, "draft_attn": 6, "select": 7, "tree": 8, "verify_attn": 9, "accept": 10,
             "commit": 11, "prep": 12, "refresh": 13, "fuse": 14}

P = C.c_void_p
I = C.c_int


class EagleError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} returned {STATUS.get(code, code)}")
        self.code = code
        self.name = STATUS.get(code, str(code))


class eagle_dims(C.Structure):
    _fields_ = [("d", I), ("n_q_heads", I), ("n_kv_heads", I), ("head_dim", I), ("d_ff", I),
                ("vocab", I), ("rms_eps", C.c_float), ("rope_theta", C.c_float)]


class eagle_limits(C.Structure):
    _fields_ = [("max_batch", I), ("max_rows", I), ("max_expanded", I), ("max_children", I),
                ("max_tree", I), ("max_prefix", I)]


class eagle_plan(C.Structure):
    _fields_ = [("kind", I), ("top_k", I), ("depth", I), ("top_m", I), ("n_expanded", I), ("n_layers", I),
                ("layer_e0", I * EAGLE_MAX_NODES), ("layer_rows", I * EAGLE_MAX_NODES), ("n_nodes", I),
                ("node_parent", C.c_int16 * EAGLE_MAX_NODES), ("node_rank", C.c_int16 * EAGLE_MAX_NODES),
                ("node_depth", C.c_int16 * EAGLE_MAX_NODES), ("node_exp", C.c_int16 * EAGLE_MAX_NODES)]


class eagle_draft_weights(C.Structure):
    _fields_ = [("w_fc", P), ("ld_fc", I), ("b_fc", P), ("g1", P), ("wq", P), ("ld_q", I), ("wk", P),
                ("ld_k", I), ("wv", P), ("ld_v", I), ("wo", P), ("ld_o", I), ("g2", P), ("w_gate", P),
                ("ld_gate", I), ("w_up", P), ("ld_up", I), ("w_down", P), ("ld_down", I), ("embed", P),
                ("ld_embed", I), ("w_lm", P), ("ld_lm", I)]


class eagle_paging(C.Structure):
    _fields_ = [("block_table", P), ("block_size", I), ("n_blocks", I)]


class eagle_kv(C.Structure):
    _fields_ = [("k", P), ("v", P), ("cap", I), ("len", P), ("paging", eagle_paging)]


class eagle_requests(C.Structure):
    _fields_ = [("t_next", P), ("f_last", P), ("pos0", P)]


class eagle_sampling(C.Structure):
    _fields_ = [("temperature", P), ("seed", C.c_uint32), ("round_id", C.c_uint32)]


class eagle_pool(C.Structure):
    _fields_ = [("token", P), ("parent", P), ("rank", P), ("depth", P), ("value", P), ("anc", P),
                ("child_exp", P)]


class eagle_children(C.Structure):
    _fields_ = [("token", P), ("prob", P)]


class eagle_draft_out(C.Structure):
    _fields_ = [("f_hat", P), ("logits", P), ("probs", P), ("k_tree", P), ("v_tree", P)]


class eagle_tree(C.Structure):
    _fields_ = [("token", P), ("parent", P), ("depth", P), ("pos", P), ("exp", P), ("anc", P),
                ("child_slot", P), ("size", P), ("stride", I)]


class eagle_accept_out(C.Structure):
    _fields_ = [("accept_len", P), ("path", P), ("final_token", P), ("last_slot", P), ("path_cap", I)]


class eagle_commit_out(C.Structure):
    _fields_ = [("f_commit", P), ("tok_commit", P), ("f_last", P), ("t_next", P), ("prefix_len", P),
                ("draft_len", P)]


_lib = None


def lib() -> C.CDLL:
    """The loaded library.  Raises if libeagle.so is missing: there is no
    fallback implementation."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libeagle.so not built ({LIB_PATH}); run "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        _lib = C.CDLL(LIB_PATH)
        _declare(_lib)
    return _lib


def _declare(L):
    s = C.c_int
    sig = {
        "eagle_create": [C.POINTER(P), C.POINTER(eagle_dims), C.POINTER(eagle_limits), C.POINTER(C.c_size_t)],
        "eagle_destroy": [P],
        "eagle_workspace_init": [P, P, P],
        "eagle_read_device_status": [P, P, P, C.POINTER(I)],
        "eagle_plan_eagle2": [C.POINTER(eagle_plan), I, I, I],
        "eagle_plan_static": [C.POINTER(eagle_plan), I, P, P],
        "eagle_draft_step": [P, C.POINTER(eagle_plan), I, I, C.POINTER(eagle_draft_weights),
                             C.POINTER(eagle_requests), C.POINTER(eagle_kv), C.POINTER(eagle_pool),
                             C.POINTER(eagle_draft_out), C.POINTER(eagle_children), C.POINTER(eagle_sampling),
                             P, P],
        "eagle_tree_expand_rerank": [P, C.POINTER(eagle_plan), I, I, I, C.POINTER(eagle_requests),
                                     C.POINTER(eagle_children), C.POINTER(eagle_pool), C.POINTER(eagle_tree),
                                     P, P],
        "eagle_tree_verify_attn": [P, I, P, P, P, C.POINTER(eagle_kv), C.POINTER(eagle_tree), C.c_float, P, P, P],
        "eagle_tree_verify_attn_noalloc": [P, I, P, P, P, C.POINTER(eagle_kv), C.POINTER(eagle_tree), C.c_float,
                                           P, P],
        "eagle_accept": [P, C.POINTER(eagle_plan), I, C.POINTER(eagle_tree), C.POINTER(eagle_children), P, P,
                         C.POINTER(eagle_sampling), P, P, C.POINTER(eagle_accept_out), P, P],
        "eagle_accept_from_probs": [P, C.POINTER(eagle_plan), I, C.POINTER(eagle_tree),
                                    C.POINTER(eagle_children), P, P, P, C.POINTER(eagle_sampling),
                                    C.POINTER(eagle_accept_out), P, P],
        "eagle_commit": [P, I, C.POINTER(eagle_accept_out), C.POINTER(eagle_tree), P, I, P, P, P, P, I, P,
                         C.POINTER(eagle_paging), C.POINTER(eagle_draft_out), C.POINTER(eagle_kv),
                         C.POINTER(eagle_commit_out), P, P],
        "eagle_trace_enable": [P, I, I],
        "eagle_trace_read": [P, C.POINTER(C.c_float), C.POINTER(I), I, C.POINTER(I)],
        "eagle_trace_disable": [P],
        "eagle_stamps_enable": [P, P, I],
        "eagle_fuse_features": [P, P, I, P, I, P, P, P, P],
        "eagle_draft_refresh": [P, I, C.POINTER(eagle_draft_weights), C.POINTER(eagle_accept_out),
                                C.POINTER(eagle_commit_out), P, C.POINTER(eagle_kv), P, P, P],
        "eagle_stamps_disable": [P, C.POINTER(I), I, C.POINTER(I)],
        "eagle_wait_selftest": [P, P, P],
    }
    for name, args in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = s
    L.eagle_status_string.argtypes = [I]
    L.eagle_status_string.restype = C.c_char_p
    L.eagle_launch_count.argtypes = [P]
    L.eagle_launch_count.restype = C.c_longlong


EXPORTED = ["eagle_create", "eagle_destroy", "eagle_workspace_init", "eagle_read_device_status",
            "eagle_status_string", "eagle_plan_eagle2", "eagle_plan_static", "eagle_draft_step",
            "eagle_tree_expand_rerank", "eagle_tree_verify_attn", "eagle_tree_verify_attn_noalloc",
            "eagle_accept", "eagle_accept_from_probs",
            "eagle_commit", "eagle_trace_enable", "eagle_trace_read", "eagle_trace_disable",
            "eagle_stamps_enable", "eagle_stamps_disable", "eagle_draft_refresh", "eagle_fuse_features",
            "eagle_launch_count", "eagle_wait_selftest"]


def _check(name: str, code: int):
    if code != 0:
        raise EagleError(name, code)


def _ref(x):
    return C.byref(x) if x is not None else None


# ---- thin wrappers with the C names -----------------------------------------

def eagle_create(dims: eagle_dims, limits: eagle_limits):
    ctx = P()
    ws = C.c_size_t()
    _check("eagle_create", lib().eagle_create(C.byref(ctx), C.byref(dims), C.byref(limits), C.byref(ws)))
    return ctx, ws.value


def eagle_destroy(ctx):
    _check("eagle_destroy", lib().eagle_destroy(ctx))


def eagle_workspace_init(ctx, ws_ptr: int, stream: int):
    _check("eagle_workspace_init", lib().eagle_workspace_init(ctx, ws_ptr, stream))


def eagle_read_device_status(ctx, ws_ptr: int, stream: int) -> int:
    v = I()
    _check("eagle_read_device_status", lib().eagle_read_device_status(ctx, ws_ptr, stream, C.byref(v)))
    return v.value


def eagle_wait_selftest(ctx, ws_ptr: int, stream: int):
    _check("eagle_wait_selftest", lib().eagle_wait_selftest(ctx, ws_ptr, stream))


def eagle_status_string(code: int) -> str:
    return lib().eagle_status_string(code).decode()


def eagle_plan_eagle2(top_k: int, depth: int, top_m: int) -> eagle_plan:
    p = eagle_plan()
    _check("eagle_plan_eagle2", lib().eagle_plan_eagle2(C.byref(p), top_k, depth, top_m))
    return p


def eagle_plan_static(parents, ranks) -> eagle_plan:
    n = len(parents)
    par = (C.c_int16 * max(n, 1))(*parents)
    rk = (C.c_int16 * max(n, 1))(*ranks)
    p = eagle_plan()
    _check("eagle_plan_static", lib().eagle_plan_static(C.byref(p), n, C.cast(par, P), C.cast(rk, P)))
    return p


def eagle_draft_step(ctx, plan, layer, batch, w, req, draft_kv, pool, out, children, s, ws_ptr, stream):
    _check("eagle_draft_step", lib().eagle_draft_step(ctx, C.byref(plan), layer, batch, C.byref(w), C.byref(req),
                                                      C.byref(draft_kv), C.byref(pool), C.byref(out),
                                                      C.byref(children), C.byref(s), ws_ptr, stream))


def eagle_tree_expand_rerank(ctx, plan, phase, layer, batch, req, children, pool, tree, ws_ptr, stream):
    _check("eagle_tree_expand_rerank",
           lib().eagle_tree_expand_rerank(ctx, C.byref(plan), phase, layer, batch, C.byref(req), _ref(children),
                                          C.byref(pool), _ref(tree), ws_ptr, stream))


def eagle_tree_verify_attn(ctx, batch, q, k_tree, v_tree, prefix, tree, scale, out, ws_ptr, stream):
    _check("eagle_tree_verify_attn",
           lib().eagle_tree_verify_attn(ctx, batch, q, k_tree, v_tree, C.byref(prefix), C.byref(tree), scale, out,
                                        ws_ptr, stream))


def eagle_tree_verify_attn_noalloc(ctx, batch, q, k_tree, v_tree, prefix, tree, scale, out, stream):
    """eagle_tree_verify_attn with its scratch in the library's fixed device
    array (no workspace); see the C header for the size limit and races."""
    _check("eagle_tree_verify_attn_noalloc",
           lib().eagle_tree_verify_attn_noalloc(ctx, batch, q, k_tree, v_tree, C.byref(prefix), C.byref(tree), scale,
                                                out, stream))


def eagle_accept(ctx, plan, batch, tree, children, target_logits, q_probs, s, target_probs, target_argmax, out,
                 ws_ptr, stream):
    _check("eagle_accept",
           lib().eagle_accept(ctx, C.byref(plan), batch, C.byref(tree), C.byref(children), target_logits, q_probs,
                              C.byref(s), target_probs, target_argmax, C.byref(out), ws_ptr, stream))


def eagle_accept_from_probs(ctx, plan, batch, tree, children, target_probs, target_argmax, q_probs, s, out,
                            ws_ptr, stream):
    _check("eagle_accept_from_probs",
           lib().eagle_accept_from_probs(ctx, C.byref(plan), batch, C.byref(tree), C.byref(children), target_probs,
                                         target_argmax, q_probs, C.byref(s), C.byref(out), ws_ptr, stream))


def eagle_commit(ctx, batch, acc, tree, f_true, k_tree_layers, v_tree_layers, k_cache_layers, v_cache_layers,
                 kv_cap, target_kv_len, draft, draft_kv, out, ws_ptr, stream, target_paging=None):
    n = len(k_tree_layers)
    arr = lambda xs: (P * max(n, 1))(*xs)
    _check("eagle_commit",
           lib().eagle_commit(ctx, batch, C.byref(acc), C.byref(tree), f_true, n, C.cast(arr(k_tree_layers), P),
                              C.cast(arr(v_tree_layers), P), C.cast(arr(k_cache_layers), P),
                              C.cast(arr(v_cache_layers), P), kv_cap, target_kv_len, _ref(target_paging),
                              _ref(draft), _ref(draft_kv), C.byref(out), ws_ptr, stream))


def eagle_fuse_features(ctx, w_fuse, ld_fuse, b_fuse, n_rows, lmh, g_out, ws_ptr, stream):
    _check("eagle_fuse_features",
           lib().eagle_fuse_features(ctx, w_fuse, ld_fuse, b_fuse or None, n_rows, lmh, g_out, ws_ptr, stream))


def eagle_draft_refresh(ctx, batch, w, acc, cm, pos0, draft_kv, len_out, ws_ptr, stream):
    _check("eagle_draft_refresh",
           lib().eagle_draft_refresh(ctx, batch, C.byref(w), C.byref(acc), C.byref(cm), pos0, C.byref(draft_kv),
                                     len_out, ws_ptr, stream))


def eagle_trace_enable(ctx, kernel: str, capacity: int):
    _check("eagle_trace_enable", lib().eagle_trace_enable(ctx, KERNEL_ID[kernel], capacity))


def eagle_trace_read(ctx, cap: int):
    """[(kernel class name, ms)] of the recorded launches, in launch order."""
    buf = (C.c_float * cap)()
    ids = (I * cap)()
    n = I()
    _check("eagle_trace_read", lib().eagle_trace_read(ctx, buf, ids, cap, C.byref(n)))
    names = {v: k for k, v in KERNEL_ID.items()}
    return [(names.get(ids[i], str(ids[i])), buf[i]) for i in range(n.value)]


def eagle_trace_disable(ctx):
    _check("eagle_trace_disable", lib().eagle_trace_disable(ctx))


def eagle_stamps_enable(ctx, stamps_ptr: int, capacity: int):
    _check("eagle_stamps_enable", lib().eagle_stamps_enable(ctx, stamps_ptr, capacity))


def eagle_stamps_disable(ctx, cap: int = 4096):
    """Kernel class names of the stamped launches, in launch order."""
    ids = (I * cap)()
    n = I()
    _check("eagle_stamps_disable", lib().eagle_stamps_disable(ctx, ids, cap, C.byref(n)))
    names = {v: k for k, v in KERNEL_ID.items()}
    return [names.get(ids[i], str(ids[i])) for i in range(min(n.value, cap))]


def eagle_launch_count(ctx) -> int:
    return int(lib().eagle_launch_count(ctx))
