"""GB300 tree-verify hot path for EAGLE-2-style speculative decoding (Python binding).

Thin ctypes binding over ``libtreespec.so`` (C ABI in ``include/treespec.h``).  The
functions below only check tensor metadata, allocate outputs with torch and pass raw
device pointers plus torch's current CUDA stream; every step of the computation runs in
the library's CUDA kernels.  There is no CPU fallback: without the built library, or
without a CUDA device, every call raises.

    tree_build(draft_logp, root_tokens, k, depth, m)      -> dict(tokens, parents, depth, mask, values)
    tree_attention(q, k_cache, v_cache, block_table, prefix_len, mask, ...) -> (out, lse)
    tree_accept(logits, tokens, parents)                  -> dict(argmax, accept_len, accept_path, bonus)

The rows after the path: ``kv_commit`` (keep the accepted path's K/V rows, release the
rejected pages), ``lm_head_argmax`` / ``tree_accept_hidden`` (target LM head with the argmax in
its GEMM epilogue), ``efficient_head`` / ``tree_build_from_topk`` (the draft's two-stage head
and the tree from its lists), ``tree_accept_sample`` (acceptance at temperature T > 0) and
``tree_prune`` (cost-aware pruning before verification).
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Dict, Optional

import torch

__all__ = [
    "TreeSpecError", "library", "library_path", "launch_count", "status_string",
    "tree_build", "tree_attention", "tree_accept", "kv_commit", "lm_head_argmax", "tree_accept_hidden",
    "efficient_head", "tree_build_from_topk", "tree_accept_sample", "tree_prune",
    "new_status", "check_status",
    "tree_build_workspace", "tree_attention_workspace", "tree_accept_workspace", "tree_attention_plan",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_PKG, "libtreespec.so")

TS_F32, TS_BF16 = 0, 1
_lib = None
_lock = threading.Lock()


class TreeSpecError(RuntimeError):
    pass


def library():
    """Load libtreespec.so (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(library_path):
            raise TreeSpecError(f"{library_path} is missing: build it with "
                                "`python -m speculative_decoding_tree_eagle_gb300.build`")
        L = ctypes.CDLL(library_path)
        P, I, S, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
        L.ts_status_string.restype = ctypes.c_char_p
        L.ts_status_string.argtypes = [I]
        L.ts_version.restype = I
        L.ts_launch_count.restype = ctypes.c_uint64
        L.ts_tree_build_workspace.restype = S
        L.ts_tree_build_workspace.argtypes = [I, I, I, I, I]
        L.ts_tree_build.restype = I
        L.ts_tree_build.argtypes = [P, P, I, I, I, I, I, P, P, P, P, P, P, P, S, P, P]
        L.ts_tree_attention_workspace.restype = S
        L.ts_tree_attention_workspace.argtypes = [I, I, I, I, I, I, I]
        L.ts_tree_attention.restype = I
        L.ts_tree_attention.argtypes = [P, P, P, I, I, I, P, I, P, I, P, I, I, I, I, I, F, P, P, P, S, P, P]
        L.ts_tree_attention_plan.restype = I
        L.ts_tree_attention_plan.argtypes = [I, I, I, I, I, I, I, I, P]
        L.ts_tree_attention_plan_for_sms.restype = I
        L.ts_tree_attention_plan_for_sms.argtypes = [I, I, I, I, I, I, I, I, I, P]
        L.ts_tree_accept_workspace.restype = S
        L.ts_tree_accept_workspace.argtypes = [I, I, I, I]
        L.ts_tree_accept.restype = I
        L.ts_tree_accept.argtypes = [P, I, P, P, I, I, I, P, P, P, P, P, S, P, P]
        L.ts_lm_head_argmax_workspace.restype = S
        L.ts_lm_head_argmax_workspace.argtypes = [I, I, I]
        L.ts_lm_head_argmax.restype = I
        L.ts_lm_head_argmax.argtypes = [P, P, I, I, I, P, P, P, S, P, P]
        L.ts_tree_accept_hidden_workspace.restype = S
        L.ts_tree_accept_hidden_workspace.argtypes = [I, I, I, I]
        L.ts_tree_accept_hidden.restype = I
        L.ts_tree_accept_hidden.argtypes = [P, P, P, P, I, I, I, I, P, P, P, P, P, S, P, P]
        L.ts_efficient_head_candidates.restype = I
        L.ts_efficient_head_candidates.argtypes = [I, I, I]
        L.ts_efficient_head_workspace.restype = S
        L.ts_efficient_head_workspace.argtypes = [I, I, I, I, I, I]
        L.ts_efficient_head.restype = I
        L.ts_efficient_head.argtypes = [P, P, P, P, I, I, I, I, I, I, I, P, P, P, P, S, P, P]
        L.ts_tree_build_from_topk.restype = I
        L.ts_tree_build_from_topk.argtypes = [P, P, P, I, I, I, I, P, P, P, P, P, P, P, P]
        L.ts_tree_accept_sample_workspace.restype = S
        L.ts_tree_accept_sample_workspace.argtypes = [I, I, I]
        L.ts_tree_accept_sample.restype = I
        L.ts_tree_accept_sample.argtypes = [P, I, P, P, P, P, P, I, I, I, I, F, I, P, P, P, P, S, P, P]
        L.ts_tree_prune_workspace.restype = S
        L.ts_tree_prune_workspace.argtypes = [I, I]
        L.ts_tree_prune.restype = I
        D = ctypes.c_double
        L.ts_tree_prune.argtypes = [P, P, P, P, P, I, I, D, D, D, P, P, P, P, P, P, P, P, P, P, S, P, P]
        L.ts_selftest_bounded_wait.restype = I
        L.ts_selftest_bounded_wait.argtypes = [I, P, P, P]
        L.ts_kv_commit.restype = I
        L.ts_kv_commit.argtypes = [P, P, I, I, I, I, I, P, I, P, P, P, I, I, P, P, P, P]
        _lib = L
    return _lib


def status_string(code: int) -> str:
    return library().ts_status_string(int(code)).decode()


def launch_count() -> int:
    """Kernels launched by the library in this process so far."""
    return int(library().ts_launch_count())


def _check(rc: int) -> None:
    if rc != 0:
        raise TreeSpecError(status_string(rc))


def _p(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def _need_cuda(name: str, t: torch.Tensor, dtype=None) -> None:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return TS_F32
    if t.dtype == torch.bfloat16:
        return TS_BF16
    raise ValueError(f"unsupported dtype {t.dtype} (fp32 or bf16)")


_ws_cache: Dict[int, torch.Tensor] = {}


def _workspace(nbytes: int, device: torch.device, ws: Optional[torch.Tensor]) -> torch.Tensor:
    if ws is not None:
        if ws.numel() * ws.element_size() < nbytes:
            raise ValueError("workspace too small")
        return ws
    idx = device.index if device.index is not None else torch.cuda.current_device()
    cur = _ws_cache.get(idx)
    if cur is None or cur.numel() < nbytes:
        cur = torch.empty(max(nbytes, 1 << 20), dtype=torch.uint8, device=device)
        _ws_cache[idx] = cur
    return cur


def new_status(device=None) -> torch.Tensor:
    """A zeroed int32 device word for the kernels' device-side error codes."""
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")


def check_status(status: torch.Tensor) -> None:
    """Synchronise and raise if a kernel reported a device-side error."""
    code = int(status.item())
    if code != 0:
        raise TreeSpecError(status_string(code))


def tree_build_workspace(B: int, V: int, k: int, depth: int, m: int) -> int:
    return int(library().ts_tree_build_workspace(B, V, k, depth, m))


def tree_attention_workspace(dtype: torch.dtype, B: int, m: int, Hq: int, Hkv: int, d: int,
                             max_prefix: int) -> int:
    dt = TS_F32 if dtype == torch.float32 else TS_BF16
    return int(library().ts_tree_attention_workspace(dt, B, m, Hq, Hkv, d, max_prefix))


def tree_attention_plan(dtype: torch.dtype, B: int, m: int, Hq: int, Hkv: int, d: int, max_prefix: int,
                        block_size: int, num_sms: Optional[int] = None) -> Dict[str, int]:
    """The launch plan tree_attention uses for these sizes on the current device, or, with
    ``num_sms``, for that many SMs (multicast and the in-cluster merge still depend on what the
    current device can co-schedule; with no device present neither is chosen)."""
    dt = TS_F32 if dtype == torch.float32 else TS_BF16
    out = (ctypes.c_int * 6)()
    if num_sms is None:
        _check(library().ts_tree_attention_plan(dt, B, m, Hq, Hkv, d, max_prefix, block_size, out))
    else:
        _check(library().ts_tree_attention_plan_for_sms(dt, B, m, Hq, Hkv, d, max_prefix, block_size,
                                                        int(num_sms), out))
    modes = {0: "one chunk", 1: "cluster merge", 2: "workspace merge"}
    return {"path": "tensor-core" if out[0] else "cuda-core", "row_groups": out[1], "chunks": out[2],
            "tiles_per_chunk": out[3], "split": modes.get(out[4], str(out[4])), "multicast": out[5]}


def tree_accept_workspace(dtype: torch.dtype, B: int, m: int, V: int) -> int:
    dt = TS_F32 if dtype == torch.float32 else TS_BF16
    return int(library().ts_tree_accept_workspace(dt, B, m, V))


def tree_build(draft_logp: torch.Tensor, root_tokens: torch.Tensor, k: int, depth: int, m: int, *,
               out: Optional[Dict[str, torch.Tensor]] = None, with_values: bool = True,
               workspace: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None) -> Dict[str, torch.Tensor]:
    """EAGLE-2 dynamic draft tree: draft_logp [B, 1+(depth-1)k, V] fp32 log-probs, root_tokens [B] int32."""
    L = library()
    _need_cuda("draft_logp", draft_logp, torch.float32)
    _need_cuda("root_tokens", root_tokens, torch.int32)
    B, R, V = draft_logp.shape
    if R != 1 + (depth - 1) * k:
        raise ValueError(f"draft_logp must have {1 + (depth - 1) * k} rows per sequence, got {R}")
    dev = draft_logp.device
    W = (m + 63) // 64
    if out is None:
        out = dict(tokens=torch.empty(B, m, dtype=torch.int32, device=dev),
                   parents=torch.empty(B, m, dtype=torch.int32, device=dev),
                   depth=torch.empty(B, m, dtype=torch.int32, device=dev),
                   mask=torch.empty(B, m, W, dtype=torch.int64, device=dev))
        if with_values:
            out["values"] = torch.empty(B, m, dtype=torch.float64, device=dev)
        out["node_row"] = torch.empty(B, m, dtype=torch.int32, device=dev)
    need = L.ts_tree_build_workspace(B, V, k, depth, m)
    if need == 0:
        raise TreeSpecError("invalid tree_build sizes")
    ws = _workspace(need, dev, workspace)
    _check(L.ts_tree_build(_p(draft_logp), _p(root_tokens), B, V, k, depth, m, _p(out["tokens"]),
                           _p(out["parents"]), _p(out["depth"]), _p(out["mask"]), _p(out.get("values")),
                           _p(out.get("node_row")), _p(ws), ws.numel() * ws.element_size(), _p(status), _stream()))
    return out


def tree_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_table: torch.Tensor,
                   prefix_len: torch.Tensor, mask: torch.Tensor, *, max_prefix: int,
                   scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                   lse: Optional[torch.Tensor] = None, with_lse: bool = True,
                   workspace: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None):
    """Tree attention.  q [B,m,Hq,d]; caches [num_blocks,Hkv,block_size,d]; block_table [B,max_blocks]
    int32; prefix_len [B] int32; mask [B,m,ceil(m/64)] (int64 view of uint64 words)."""
    L = library()
    for name, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache)):
        _need_cuda(name, t, q.dtype)
    _need_cuda("block_table", block_table, torch.int32)
    _need_cuda("prefix_len", prefix_len, torch.int32)
    _need_cuda("mask", mask, torch.int64)
    B, m, Hq, d = q.shape
    NB, Hkv, bs, d2 = k_cache.shape
    if d2 != d or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("cache shapes do not match q")
    if mask.shape != (B, m, (m + 63) // 64):
        raise ValueError("mask must be [B, m, ceil(m/64)]")
    dt = _dt(q)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and with_lse:
        lse = torch.empty(B, m, Hq, dtype=torch.float32, device=q.device)
    need = L.ts_tree_attention_workspace(dt, B, m, Hq, Hkv, d, max_prefix)
    ws = _workspace(max(need, 256), q.device, workspace)
    _check(L.ts_tree_attention(_p(q), _p(k_cache), _p(v_cache), dt, NB, bs, _p(block_table),
                               block_table.shape[1], _p(prefix_len), int(max_prefix), _p(mask), B, m, Hq,
                               Hkv, d, float(scale), _p(out), _p(lse), _p(ws),
                               ws.numel() * ws.element_size(), _p(status), _stream()))
    return out, lse


def tree_accept(logits: torch.Tensor, tokens: torch.Tensor, parents: torch.Tensor, *,
                out: Optional[Dict[str, torch.Tensor]] = None, workspace: Optional[torch.Tensor] = None,
                status: Optional[torch.Tensor] = None) -> Dict[str, torch.Tensor]:
    """Per-node argmax of logits [B,m,V] and the longest matching root path."""
    L = library()
    _need_cuda("logits", logits)
    _need_cuda("tokens", tokens, torch.int32)
    _need_cuda("parents", parents, torch.int32)
    B, m, V = logits.shape
    dt = _dt(logits)
    dev = logits.device
    if out is None:
        out = dict(argmax=torch.empty(B, m, dtype=torch.int32, device=dev),
                   accept_len=torch.empty(B, dtype=torch.int32, device=dev),
                   accept_path=torch.empty(B, m, dtype=torch.int32, device=dev),
                   bonus=torch.empty(B, dtype=torch.int32, device=dev))
    need = L.ts_tree_accept_workspace(dt, B, m, V)
    if need == 0:
        raise TreeSpecError("invalid tree_accept sizes")
    ws = _workspace(need, dev, workspace)
    _check(L.ts_tree_accept(_p(logits), dt, _p(tokens), _p(parents), B, m, V, _p(out["argmax"]),
                            _p(out["accept_len"]), _p(out["accept_path"]), _p(out["bonus"]), _p(ws),
                            ws.numel() * ws.element_size(), _p(status), _stream()))
    return out


Q_MODES = {"point": 0, "draft": 1}


def tree_accept_sample(logits: torch.Tensor, tokens: torch.Tensor, parents: torch.Tensor, uniforms: torch.Tensor,
                       temperature: float, *, q_mode: str = "point", draft_logp: Optional[torch.Tensor] = None,
                       node_row: Optional[torch.Tensor] = None, out: Optional[Dict[str, torch.Tensor]] = None,
                       workspace: Optional[torch.Tensor] = None,
                       status: Optional[torch.Tensor] = None) -> Dict[str, torch.Tensor]:
    """Verification at temperature T > 0 by multi-round rejection sampling: logits [B,m,V],
    tokens/parents [B,m] int32, uniforms [B,m] float32 in [0, 1).  q_mode "point" (a unit mass
    per candidate) or "draft" (the draft rows draft_logp [B,R,V] named by node_row [B,m]).
    Returns accept_len [B], accept_path [B,m] and bonus [B] (the drawn token)."""
    L = library()
    _need_cuda("logits", logits)
    _need_cuda("tokens", tokens, torch.int32)
    _need_cuda("parents", parents, torch.int32)
    _need_cuda("uniforms", uniforms, torch.float32)
    if q_mode not in Q_MODES:
        raise TreeSpecError("q_mode is 'point' or 'draft'")
    B, m, V = logits.shape
    R = 0
    if q_mode == "draft":
        if draft_logp is None or node_row is None:
            raise TreeSpecError("q_mode 'draft' needs draft_logp and node_row")
        _need_cuda("draft_logp", draft_logp, torch.float32)
        _need_cuda("node_row", node_row, torch.int32)
        R = draft_logp.shape[1]
    dev = logits.device
    if out is None:
        out = dict(accept_len=torch.empty(B, dtype=torch.int32, device=dev),
                   accept_path=torch.empty(B, m, dtype=torch.int32, device=dev),
                   bonus=torch.empty(B, dtype=torch.int32, device=dev))
    need = L.ts_tree_accept_sample_workspace(B, V, Q_MODES[q_mode])
    ws = _workspace(need, dev, workspace) if need > 0 else None
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(L.ts_tree_accept_sample(_p(logits), _dt(logits), _p(tokens), _p(parents), _p(uniforms), _p(draft_logp),
                                   _p(node_row), R, B, m, V, float(temperature), Q_MODES[q_mode],
                                   _p(out["accept_len"]), _p(out["accept_path"]), _p(out["bonus"]), _p(ws), nbytes,
                                   _p(status), _stream()))
    return out


def tree_prune(tree: Dict[str, torch.Tensor], t_draft: float, t_fixed: float, t_node: float, *,
               workspace: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
               sync: bool = True) -> Dict[str, torch.Tensor]:
    """Cost-aware pruning before verification of a tree from tree_build (``tokens``, ``parents``,
    ``depth`` int32 and ``values`` float64 [B,m]; ``node_row`` optional).  One node count n for
    the batch maximises expected tokens per unit of round time (t_draft + t_fixed + t_node*B*n).
    Returns ``n`` (a device int32 [1]) and the pruned tree: ``tokens``, ``parents``, ``depth``,
    ``kept`` (old flat indices), ``node_row`` int32 and ``values`` [B,n], ``mask`` int64
    [B,n,ceil(n/64)], ``expected`` float32 [B].  With ``sync`` (default) the host reads n and
    the outputs are views of shape [B,n]; without it they are the flat buffers (row stride n)."""
    L = library()
    for name, dt in (("tokens", torch.int32), ("parents", torch.int32), ("depth", torch.int32),
                     ("values", torch.float64)):
        _need_cuda(name, tree[name], dt)
    nr = tree.get("node_row")
    if nr is not None:
        _need_cuda("node_row", nr, torch.int32)
    B, m = tree["tokens"].shape
    dev = tree["tokens"].device
    W = (m + 63) // 64
    buf = dict(n=torch.empty(1, dtype=torch.int32, device=dev),
               tokens=torch.empty(B * m, dtype=torch.int32, device=dev),
               parents=torch.empty(B * m, dtype=torch.int32, device=dev),
               depth=torch.empty(B * m, dtype=torch.int32, device=dev),
               kept=torch.empty(B * m, dtype=torch.int32, device=dev),
               values=torch.empty(B * m, dtype=torch.float64, device=dev),
               mask=torch.empty(B * m * W, dtype=torch.int64, device=dev),
               expected=torch.empty(B, dtype=torch.float32, device=dev))
    if nr is not None:
        buf["node_row"] = torch.empty(B * m, dtype=torch.int32, device=dev)
    need = L.ts_tree_prune_workspace(B, m)
    if need == 0:
        raise TreeSpecError("invalid tree_prune sizes")
    ws = _workspace(need, dev, workspace)
    _check(L.ts_tree_prune(_p(tree["tokens"]), _p(tree["parents"]), _p(tree["depth"]), _p(tree["values"]), _p(nr),
                           B, m, float(t_draft), float(t_fixed), float(t_node), _p(buf["n"]), _p(buf["tokens"]),
                           _p(buf["parents"]), _p(buf["depth"]), _p(buf["mask"]), _p(buf["values"]),
                           _p(buf.get("node_row")), _p(buf["kept"]), _p(buf["expected"]), _p(ws),
                           ws.numel() * ws.element_size(), _p(status), _stream()))
    if not sync:
        return buf
    n = int(buf["n"].item())
    Wn = (n + 63) // 64
    out = {"n": buf["n"], "expected": buf["expected"]}
    for k in ("tokens", "parents", "depth", "kept", "values", "node_row"):
        if k in buf:
            out[k] = buf[k][: B * n].view(B, n)
    out["mask"] = buf["mask"][: B * n * Wn].view(B, n, Wn)
    return out


def kv_commit(k_cache: torch.Tensor, v_cache: torch.Tensor, block_table: torch.Tensor,
              prefix_len: torch.Tensor, accept_path: torch.Tensor, accept_len: torch.Tensor, *,
              out: Optional[Dict[str, torch.Tensor]] = None,
              status: Optional[torch.Tensor] = None) -> Dict[str, torch.Tensor]:
    """Keep the accepted path's K/V rows and release the rejected scratch pages, in place on
    k_cache/v_cache [num_blocks,Hkv,bs,d], block_table [B,max_blocks] and prefix_len [B];
    returns freed_blocks [B,max_blocks] (-1 padded) and freed_count [B]."""
    L = library()
    _need_cuda("k_cache", k_cache)
    _need_cuda("v_cache", v_cache, k_cache.dtype)
    _need_cuda("block_table", block_table, torch.int32)
    _need_cuda("prefix_len", prefix_len, torch.int32)
    _need_cuda("accept_path", accept_path, torch.int32)
    _need_cuda("accept_len", accept_len, torch.int32)
    nb, hkv, bs, d = k_cache.shape
    B, max_blocks = block_table.shape
    m = accept_path.shape[1]
    dev = k_cache.device
    if out is None:
        out = dict(freed_blocks=torch.empty(B, max_blocks, dtype=torch.int32, device=dev),
                   freed_count=torch.empty(B, dtype=torch.int32, device=dev))
    _check(L.ts_kv_commit(_p(k_cache), _p(v_cache), _dt(k_cache), nb, bs, hkv, d, _p(block_table), max_blocks,
                          _p(prefix_len), _p(accept_path), _p(accept_len), B, m, _p(out["freed_blocks"]),
                          _p(out["freed_count"]), _p(status), _stream()))
    return out


def lm_head_argmax(hidden: torch.Tensor, weight: torch.Tensor, *, out: Optional[Dict[str, torch.Tensor]] = None,
                   workspace: Optional[torch.Tensor] = None,
                   status: Optional[torch.Tensor] = None) -> Dict[str, torch.Tensor]:
    """Per-row argmax (first index) and max of hidden [M,K] @ weight[N,K]^T (bf16), logits kept on chip."""
    L = library()
    _need_cuda("hidden", hidden, torch.bfloat16)
    _need_cuda("weight", weight, torch.bfloat16)
    M, K = hidden.shape
    N, K2 = weight.shape
    if K2 != K:
        raise ValueError("hidden and weight disagree on K")
    dev = hidden.device
    if out is None:
        out = dict(argmax=torch.empty(M, dtype=torch.int32, device=dev),
                   max_logit=torch.empty(M, dtype=torch.float32, device=dev))
    need = L.ts_lm_head_argmax_workspace(M, N, K)
    if need == 0:
        raise TreeSpecError("invalid lm_head_argmax sizes")
    ws = _workspace(need, dev, workspace)
    _check(L.ts_lm_head_argmax(_p(hidden), _p(weight), M, N, K, _p(out["argmax"]), _p(out.get("max_logit")), _p(ws),
                               ws.numel() * ws.element_size(), _p(status), _stream()))
    return out


def tree_accept_hidden(hidden: torch.Tensor, weight: torch.Tensor, tokens: torch.Tensor, parents: torch.Tensor, *,
                       out: Optional[Dict[str, torch.Tensor]] = None, workspace: Optional[torch.Tensor] = None,
                       status: Optional[torch.Tensor] = None) -> Dict[str, torch.Tensor]:
    """tree_accept from the target's final hidden states [B,m,K] and its LM head [V,K] (bf16)."""
    L = library()
    _need_cuda("hidden", hidden, torch.bfloat16)
    _need_cuda("weight", weight, torch.bfloat16)
    _need_cuda("tokens", tokens, torch.int32)
    _need_cuda("parents", parents, torch.int32)
    B, m, K = hidden.shape
    V = weight.shape[0]
    dev = hidden.device
    if out is None:
        out = dict(argmax=torch.empty(B, m, dtype=torch.int32, device=dev),
                   accept_len=torch.empty(B, dtype=torch.int32, device=dev),
                   accept_path=torch.empty(B, m, dtype=torch.int32, device=dev),
                   bonus=torch.empty(B, dtype=torch.int32, device=dev))
    need = L.ts_tree_accept_hidden_workspace(B, m, V, K)
    if need == 0:
        raise TreeSpecError("invalid tree_accept_hidden sizes")
    ws = _workspace(need, dev, workspace)
    _check(L.ts_tree_accept_hidden(_p(hidden), _p(weight), _p(tokens), _p(parents), B, m, V, K, _p(out["argmax"]),
                                   _p(out["accept_len"]), _p(out["accept_path"]), _p(out["bonus"]), _p(ws),
                                   ws.numel() * ws.element_size(), _p(status), _stream()))
    return out


def efficient_head(hidden: torch.Tensor, lr_b: torch.Tensor, lr_a: torch.Tensor, weight: torch.Tensor, *,
                   tile_tokens: int, k_tile: int, k: int, with_candidates: bool = False,
                   workspace: Optional[torch.Tensor] = None,
                   status: Optional[torch.Tensor] = None) -> Dict[str, torch.Tensor]:
    """Two-stage draft head: hidden [M,d], lr_b [rank,d], lr_a [V,rank], weight [V,d] (bf16) ->
    top_tok [M,k], top_logp [M,k] (log-probs over the candidates), optionally candidates [M,C]."""
    L = library()
    for n, t in (("hidden", hidden), ("lr_b", lr_b), ("lr_a", lr_a), ("weight", weight)):
        _need_cuda(n, t, torch.bfloat16)
    M, d = hidden.shape
    rank = lr_b.shape[0]
    V = weight.shape[0]
    dev = hidden.device
    C = L.ts_efficient_head_candidates(V, tile_tokens, k_tile)
    out = dict(top_tok=torch.empty(M, k, dtype=torch.int32, device=dev),
               top_logp=torch.empty(M, k, dtype=torch.float32, device=dev))
    if with_candidates:
        out["candidates"] = torch.empty(M, max(C, 1), dtype=torch.int32, device=dev)
    need = L.ts_efficient_head_workspace(M, V, d, rank, tile_tokens, k_tile)
    if need == 0:
        raise TreeSpecError("invalid efficient_head sizes")
    ws = _workspace(need, dev, workspace)
    _check(L.ts_efficient_head(_p(hidden), _p(lr_b), _p(lr_a), _p(weight), M, V, d, rank, tile_tokens, k_tile, k,
                               _p(out["top_tok"]), _p(out["top_logp"]), _p(out.get("candidates")), _p(ws),
                               ws.numel() * ws.element_size(), _p(status), _stream()))
    return out


def tree_build_from_topk(row_tok: torch.Tensor, row_logp: torch.Tensor, root_tokens: torch.Tensor, k: int,
                         depth: int, m: int, *, out: Optional[Dict[str, torch.Tensor]] = None,
                         status: Optional[torch.Tensor] = None) -> Dict[str, torch.Tensor]:
    """tree_build from per-row top-k lists row_tok [B,R,k] int32 / row_logp [B,R,k] fp32."""
    L = library()
    _need_cuda("row_tok", row_tok, torch.int32)
    _need_cuda("row_logp", row_logp, torch.float32)
    _need_cuda("root_tokens", root_tokens, torch.int32)
    B = row_tok.shape[0]
    dev = row_tok.device
    W = (m + 63) // 64
    if out is None:
        out = dict(tokens=torch.empty(B, m, dtype=torch.int32, device=dev),
                   parents=torch.empty(B, m, dtype=torch.int32, device=dev),
                   depth=torch.empty(B, m, dtype=torch.int32, device=dev),
                   mask=torch.empty(B, m, W, dtype=torch.int64, device=dev),
                   values=torch.empty(B, m, dtype=torch.float64, device=dev),
                   node_row=torch.empty(B, m, dtype=torch.int32, device=dev))
    _check(L.ts_tree_build_from_topk(_p(row_tok), _p(row_logp), _p(root_tokens), B, k, depth, m, _p(out["tokens"]),
                                     _p(out["parents"]), _p(out["depth"]), _p(out["mask"]), _p(out.get("values")),
                                     _p(out.get("node_row")), _p(status), _stream()))
    return out
