"""Python binding of libserac_gb300.so: exhaustive SIFT descriptor matching with a
fused top-2 on GB300 (sm_103a).

This module only marshals arguments for the C ABI declared in ``include/serac.h``;
every step of the matching runs in the library's CUDA kernels.  PyTorch supplies the
device memory (inputs, outputs, workspace) and the stream.  There is no fallback: if
the library is missing or the GPU is not an sm_103 part, the calls raise.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional, Sequence

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libserac_gb300.so")

OK, EINVAL, ECAPACITY, ECUDA, ETIMEOUT, EWORKSPACE, EUNSUPPORTED = 0, -1, -2, -3, -4, -5, -6
DIM = 128
NOALLOC_SCRATCH_BYTES = 16 << 20  # SERAC_NOALLOC_SCRATCH_BYTES

# every symbol include/serac.h declares
EXPORTS = ("serac_default_params", "serac_pair_workspace_size", "match_pair",
           "match_batch_workspace_size", "match_batch", "serac_scores",
           "serac_set_profile_events", "serac_device_check", "serac_last_launch_count",
           "serac_schedule_describe", "serac_status_str", "match_pair_noalloc",
           "serac_last_cuda_error", "serac_test_inject_timeout", "serac_topk_workspace_size",
           "serac_topk_pair")


class SeracError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = f"{what}: {status_str(status)} ({status})" if what else status_str(status)
        if status == ECUDA:
            msg += f" [cudaError {int(lib().serac_last_cuda_error())}]"
        super().__init__(msg)


class Params(ctypes.Structure):
    _fields_ = [("ratio_num_sq", ctypes.c_int32), ("ratio_den_sq", ctypes.c_int32),
                ("norm_sq", ctypes.c_int32), ("min_score", ctypes.c_int32),
                ("mutual", ctypes.c_int32), ("col_ratio", ctypes.c_int32),
                ("max_features", ctypes.c_int32)]

    def __repr__(self):
        return ("Params(" + ", ".join(f"{n}={getattr(self, n)}" for n, _ in self._fields_) + ")")


class _Pair(ctypes.Structure):
    _fields_ = [("a", ctypes.c_void_p), ("n_a", ctypes.c_int32),
                ("b", ctypes.c_void_p), ("n_b", ctypes.c_int32)]


class _Out(ctypes.Structure):
    _fields_ = [("matches", ctypes.c_void_p), ("capacity", ctypes.c_int32),
                ("count", ctypes.c_void_p), ("row_top2", ctypes.c_void_p),
                ("col_top2", ctypes.c_void_p)]


_lib_handle = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib_handle
    if _lib_handle is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"{_LIB_PATH} is missing: build it first "
                               "(python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(_LIB_PATH)
        P, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        L.serac_default_params.argtypes = [ctypes.POINTER(Params), ctypes.c_float, ctypes.c_float]
        L.serac_pair_workspace_size.argtypes = [i32, i32]
        L.serac_pair_workspace_size.restype = sz
        L.match_pair.argtypes = [P, i32, P, i32, ctypes.POINTER(Params), ctypes.POINTER(_Out), P, sz, P]
        L.match_batch_workspace_size.argtypes = [ctypes.POINTER(_Pair), i32]
        L.match_batch_workspace_size.restype = sz
        L.match_batch.argtypes = [ctypes.POINTER(_Pair), i32, ctypes.POINTER(Params),
                                  ctypes.POINTER(_Out), P, sz, P]
        L.serac_scores.argtypes = [P, i32, P, i32, P, P, sz, P]
        L.serac_set_profile_events.argtypes = [P, P]
        L.serac_schedule_describe.argtypes = [ctypes.POINTER(_Pair), i32, i32, P, P, P, P]
        L.serac_status_str.restype = ctypes.c_char_p
        L.match_pair_noalloc.argtypes = [P, i32, P, i32, ctypes.POINTER(Params), ctypes.POINTER(_Out), P]
        L.serac_test_inject_timeout.argtypes = [ctypes.c_int]
        L.serac_topk_workspace_size.argtypes = [i32, i32, i32]
        L.serac_topk_workspace_size.restype = sz
        L.serac_topk_pair.argtypes = [P, i32, P, i32, i32, P, P, P, P, sz, P]
        _lib_handle = L
    return _lib_handle


def status_str(status: int) -> str:
    return lib().serac_status_str(int(status)).decode()


def _check(status: int, what: str) -> None:
    if status != OK:
        raise SeracError(status, what)


def default_params(max_ratio: float = 0.8, max_angle: float = 0.7, mutual: int = 1,
                   col_ratio: int = 1, max_features: int = 0) -> Params:
    """Integer test parameters from the ratio and the maximum angle (serac_default_params);
    max_features = K > 0 matches only the first K descriptors of each image."""
    p = Params()
    _check(lib().serac_default_params(ctypes.byref(p), max_ratio, max_angle), "serac_default_params")
    p.mutual, p.col_ratio, p.max_features = int(mutual), int(col_ratio), int(max_features)
    return p


def _capped(p: Params, n: int) -> int:
    return min(n, p.max_features) if p.max_features > 0 else n


def device_check() -> int:
    return int(lib().serac_device_check())


def last_launch_count() -> int:
    return int(lib().serac_last_launch_count())


def inject_timeout(enable: bool = True) -> None:
    """Failure-detection test hook: the next call's TMA producer issues no copies, so
    its bounded waits run out (2 s) and the call reports ETIMEOUT through `count`."""
    lib().serac_test_inject_timeout(1 if enable else 0)


def set_profile_events(begin: Optional[torch.cuda.Event], end: Optional[torch.cuda.Event]) -> None:
    """Events must already exist (torch creates them on their first record)."""
    hb = begin.cuda_event if begin is not None else None
    he = end.cuda_event if end is not None else None
    if (begin is not None and not hb) or (end is not None and not he):
        raise ValueError("record the events once before handing them to the library")
    lib().serac_set_profile_events(hb, he)


def pair_workspace_size(n_a: int, n_b: int) -> int:
    return int(lib().serac_pair_workspace_size(int(n_a), int(n_b)))


def _desc(x: torch.Tensor, name: str) -> torch.Tensor:
    """CUDA tensors, or pinned host tensors (the staging kernel reads those directly
    over the host link)."""
    if x.dtype != torch.uint8 or x.dim() != 2 or x.shape[1] != DIM or not (x.is_cuda or x.is_pinned()):
        raise ValueError(f"{name}: expected a CUDA or pinned-host uint8 tensor of shape (n, {DIM})")
    if not x.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    return x


def _stream_ptr(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def workspace(nbytes: int, device) -> torch.Tensor:
    """Caller-owned device scratch (256-byte aligned by the caching allocator)."""
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


@dataclass
class MatchOutput:
    """Device outputs of one pair.  `count` holds the number of matches (or a negative
    status); `matches` has room for `capacity` rows of (i, j), ascending i."""
    matches: torch.Tensor
    count: torch.Tensor
    row_top2: Optional[torch.Tensor]
    col_top2: Optional[torch.Tensor]

    def result(self):
        """Synchronise and return the matches as a (count, 2) int32 CPU tensor."""
        if not self.count.is_cuda:  # written by the kernels into host memory
            torch.cuda.synchronize()
        n = int(self.count.item())
        if n < 0:
            raise SeracError(n, "match")
        if n > self.matches.shape[0]:
            raise SeracError(ECAPACITY, f"match ({n} matches, capacity {self.matches.shape[0]})")
        return self.matches[:n].cpu()


def _make_out(n_a: int, n_b: int, device, capacity: Optional[int], top2: bool, host: bool = False):
    cap = n_a if capacity is None else int(capacity)

    def buf(shape):
        if host:  # pinned host memory the kernels write directly
            return torch.empty(shape, dtype=torch.int32, pin_memory=True)
        return torch.empty(shape, dtype=torch.int32, device=device)

    o = MatchOutput(matches=buf((max(cap, 1), 2)), count=buf((1,)),
                    row_top2=buf((max(n_a, 1), 4)) if top2 else None,
                    col_top2=buf((max(n_b, 1), 4)) if top2 else None)
    c = _Out(o.matches.data_ptr(), cap, o.count.data_ptr(),
             o.row_top2.data_ptr() if top2 else None, o.col_top2.data_ptr() if top2 else None)
    return o, c


def output_for(o: MatchOutput):
    """The C-ABI output record of an existing MatchOutput (to reuse its buffers)."""
    return _Out(o.matches.data_ptr(), o.matches.shape[0], o.count.data_ptr(),
                o.row_top2.data_ptr() if o.row_top2 is not None else None,
                o.col_top2.data_ptr() if o.col_top2 is not None else None)


def match_pair(a: torch.Tensor, b: torch.Tensor, params: Optional[Params] = None, *,
               capacity: Optional[int] = None, top2: bool = False,
               workspace_t: Optional[torch.Tensor] = None, stream=None,
               out: Optional[MatchOutput] = None, host_out: bool = False) -> MatchOutput:
    """Match descriptors a (n_a, 128) against b (n_b, 128), asynchronously.

    a and b may be CUDA tensors or pinned host tensors.  `out` (from an earlier call
    with the same sizes) reuses its buffers; host_out=True puts new outputs in pinned
    host memory, written by the kernels directly (read them after synchronising)."""
    a, b = _desc(a, "a"), _desc(b, "b")
    p = params if params is not None else default_params()
    n_a, n_b = a.shape[0], b.shape[0]
    dev = a.device if a.is_cuda else (b.device if b.is_cuda else torch.device("cuda", torch.cuda.current_device()))
    if workspace_t is not None:
        ws = workspace_t
    else:
        ws = workspace(pair_workspace_size(n_a, n_b), dev)
    if out is not None:
        o, c = out, output_for(out)
    else:
        o, c = _make_out(_capped(p, n_a), _capped(p, n_b), dev, capacity, top2, host=host_out)
    st = lib().match_pair(a.data_ptr(), n_a, b.data_ptr(), n_b, ctypes.byref(p), ctypes.byref(c),
                          ws.data_ptr(), ws.numel(), _stream_ptr(stream))
    _check(st, "match_pair")
    return o


def match_pair_noalloc(a: torch.Tensor, b: torch.Tensor, params: Optional[Params] = None, *,
                       capacity: Optional[int] = None, top2: bool = False, stream=None) -> MatchOutput:
    """match_pair on the library's built-in scratch, for callers that may not allocate
    device memory for a workspace (see include/serac.h).  The outputs are still the
    caller's.  Calls sharing the scratch must not overlap on the GPU."""
    a, b = _desc(a, "a"), _desc(b, "b")
    p = params if params is not None else default_params()
    o, c = _make_out(_capped(p, a.shape[0]), _capped(p, b.shape[0]), a.device, capacity, top2)
    st = lib().match_pair_noalloc(a.data_ptr(), a.shape[0], b.data_ptr(), b.shape[0], ctypes.byref(p),
                                  ctypes.byref(c), _stream_ptr(stream))
    _check(st, "match_pair_noalloc")
    return o


MAX_TOPK = 8


@dataclass
class TopkOutput:
    """Row top-k of one pair: scores and index (n_a, k) int32 -- row i's k best columns,
    score descending then lower column first, padded (0, -1) -- and `status` (1,) int32:
    OK, or ETIMEOUT when a bounded wait inside a kernel ran out."""
    scores: torch.Tensor
    index: torch.Tensor
    status: torch.Tensor


def topk_workspace_size(n_a: int, n_b: int, k: int) -> int:
    """Workspace bytes of topk_pair on the current device (0 on bad arguments)."""
    return int(lib().serac_topk_workspace_size(int(n_a), int(n_b), int(k)))


def topk_pair(a: torch.Tensor, b: torch.Tensor, k: int, *, workspace_t: Optional[torch.Tensor] = None,
              stream=None, out: Optional[TopkOutput] = None, host_out: bool = False) -> TopkOutput:
    """Row top-k (guided matching candidates) of a against b, asynchronously: for every
    row of a, its k (1..8) highest-scoring rows of b.  a and b may be CUDA or pinned
    host tensors; host_out=True puts the outputs in pinned host memory."""
    a, b = _desc(a, "a"), _desc(b, "b")
    n_a, n_b = a.shape[0], b.shape[0]
    dev = a.device if a.is_cuda else (b.device if b.is_cuda else torch.device("cuda", torch.cuda.current_device()))
    if not 1 <= int(k) <= MAX_TOPK:
        raise SeracError(EINVAL, f"topk_pair (k = {k})")
    ws = workspace_t if workspace_t is not None else workspace(topk_workspace_size(n_a, n_b, k), dev)
    if out is None:
        def buf(shape):
            if host_out:
                return torch.empty(shape, dtype=torch.int32, pin_memory=True)
            return torch.empty(shape, dtype=torch.int32, device=dev)
        out = TopkOutput(scores=buf((max(n_a, 1), int(k))), index=buf((max(n_a, 1), int(k))), status=buf((1,)))
    st = lib().serac_topk_pair(a.data_ptr(), n_a, b.data_ptr(), n_b, int(k), out.scores.data_ptr(),
                               out.index.data_ptr(), out.status.data_ptr(), ws.data_ptr(), ws.numel(),
                               _stream_ptr(stream))
    _check(st, "topk_pair")
    return out


def _pairs_struct(pairs: Sequence):
    arr = (_Pair * max(len(pairs), 1))()
    for k, (a, b) in enumerate(pairs):
        _desc(a, f"pairs[{k}].a")
        _desc(b, f"pairs[{k}].b")
        arr[k] = _Pair(a.data_ptr(), a.shape[0], b.data_ptr(), b.shape[0])
    return arr


def batch_workspace_size(pairs: Sequence) -> int:
    arr = _pairs_struct(pairs)
    return int(lib().match_batch_workspace_size(arr, len(pairs)))


def match_batch(pairs: Sequence, params: Optional[Params] = None, *, capacities=None,
                top2: bool = False, workspace_t: Optional[torch.Tensor] = None,
                stream=None, outs: Optional[list] = None, host_out: bool = False) -> list:
    """Match every (a, b) of `pairs`; images shared between pairs are staged once.

    Images may be CUDA tensors or pinned host tensors.  `outs` (from an earlier call
    with the same pairs) reuses those buffers; host_out=True puts new outputs in
    pinned host memory, written by the kernels directly (read them after
    synchronising)."""
    arr = _pairs_struct(pairs)
    p = params if params is not None else default_params()
    n = len(pairs)
    if outs is not None and len(outs) != n:
        raise ValueError("outs: one MatchOutput per pair expected")
    need = int(lib().match_batch_workspace_size(arr, n))
    dev = torch.device("cuda", torch.cuda.current_device())
    for a, b in pairs:
        if a.is_cuda:
            dev = a.device
            break
    ws = workspace_t if workspace_t is not None else workspace(need, dev)
    res, couts = [], (_Out * max(n, 1))()
    for k, (a, b) in enumerate(pairs):
        if outs is not None:
            o, c = outs[k], output_for(outs[k])
        else:
            cap = None if capacities is None else capacities[k]
            o, c = _make_out(_capped(p, a.shape[0]), _capped(p, b.shape[0]), dev, cap, top2, host=host_out)
        res.append(o)
        couts[k] = c
    st = lib().match_batch(arr, n, ctypes.byref(p), couts, ws.data_ptr(), ws.numel(), _stream_ptr(stream))
    _check(st, "match_batch")
    return res


def scores(a: torch.Tensor, b: torch.Tensor, *, workspace_t: Optional[torch.Tensor] = None,
           stream=None) -> torch.Tensor:
    """Full (n_a, n_b) int32 score matrix from the same tensor-core tiles (small n)."""
    a, b = _desc(a, "a"), _desc(b, "b")
    n_a, n_b = a.shape[0], b.shape[0]
    out = torch.empty((max(n_a, 1), max(n_b, 1)), dtype=torch.int32, device=a.device)
    ws = workspace_t if workspace_t is not None else workspace(pair_workspace_size(n_a, n_b), a.device)
    st = lib().serac_scores(a.data_ptr(), n_a, b.data_ptr(), n_b, out.data_ptr(), ws.data_ptr(),
                            ws.numel(), _stream_ptr(stream))
    _check(st, "serac_scores")
    return out[:n_a, :n_b]


def shard_pairs(sizes: Sequence, world: int) -> list:
    """Split pairs with these (n_a, n_b) over `world` GPUs, one process each, by cost
    (n_a * n_b, the contraction's size): longest-processing-time greedy, each pair to
    the least-loaded rank.  Returns, per rank, the ascending indices of its pairs.
    Pairs are independent, so a rank runs match_batch on its own shard and no data
    crosses ranks; a caller that wants every result in one place gathers them after."""
    if world < 1:
        raise ValueError("world must be >= 1")
    order = sorted(range(len(sizes)), key=lambda k: (-int(sizes[k][0]) * int(sizes[k][1]), k))
    load = [0] * world
    shards = [[] for _ in range(world)]
    for k in order:
        r = min(range(world), key=lambda i: (load[i], i))
        shards[r].append(k)
        load[r] += int(sizes[k][0]) * int(sizes[k][1])
    return [sorted(x) for x in shards]


def match_batch_shard(pairs: Sequence, rank: int, world: int, params: Optional[Params] = None, **kwargs):
    """One GPU's share of a sharded batch: the pairs shard_pairs() gives `rank` of
    `world`, matched by one match_batch on the current device.  Returns (indices of
    those pairs in `pairs`, their MatchOutputs).  Nothing crosses ranks here; see
    gather_matches for collecting the lists afterwards."""
    sizes = [(int(a.shape[0]), int(b.shape[0])) for a, b in pairs]
    mine = shard_pairs(sizes, world)[rank]
    outs = match_batch([pairs[k] for k in mine], params, **kwargs) if mine else []
    return mine, outs


def gather_matches(mine: Sequence, outs: Sequence, n_pairs: int, group=None, dst: int = 0):
    """Collect the match lists of a sharded batch on rank `dst` after every rank has run
    its match_batch_shard: returns, on `dst`, the list of all n_pairs (count, 2) int32
    CPU tensors in the batch's pair order, and None on the other ranks.  A host-side
    collection (torch.distributed.gather_object over the process group), after the
    GPU work; the matching itself has no collective."""
    import torch.distributed as dist
    local = [(int(k), o.result()) for k, o in zip(mine, outs)]
    rank = dist.get_rank(group)
    parts = [None] * dist.get_world_size(group) if rank == dst else None
    dist.gather_object(local, parts, dst=dst, group=group)
    if rank != dst:
        return None
    res = [None] * n_pairs
    for part in parts:
        for k, m in part:
            if res[k] is not None:
                raise RuntimeError(f"pair {k} came from two ranks")
            res[k] = m
    missing = [k for k, m in enumerate(res) if m is None]
    if missing:
        raise RuntimeError(f"pairs {missing[:8]} came from no rank")
    return res


def schedule_describe(sizes: Sequence, grid: int):
    """Host-side view of how the first launch chunk of pairs with these (n_a, n_b)
    sizes is cut: (chunks, pieces, pieces per row problem -- two per pair: A's rows,
    then B's rows --, tiles per CTA[grid])."""
    n = len(sizes)
    arr = (_Pair * max(n, 1))()
    for k, (na, nb) in enumerate(sizes):
        arr[k] = _Pair(16 * (2 * k + 1), int(na), 16 * (2 * k + 2), int(nb))
    chunks, pieces = ctypes.c_int32(), ctypes.c_int32()
    npieces = (ctypes.c_int32 * max(2 * n, 1))()
    cta_tiles = (ctypes.c_int32 * grid)()
    _check(lib().serac_schedule_describe(arr, n, grid, ctypes.byref(chunks), ctypes.byref(pieces),
                                         npieces, cta_tiles), "serac_schedule_describe")
    return chunks.value, pieces.value, list(npieces)[:2 * n], list(cta_tiles)
