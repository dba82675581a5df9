"""ctypes binding of libtide (include/tide.h): argument marshalling only.

Every step of the hot path runs in the CUDA library; this module turns Python
shapes, torch tensors and streams into the C ABI's plain integers and
pointers.  Importing it loads ``libtide.so`` from this package directory and
raises ``TideError`` if the library is missing -- there is no fallback.

Names match the C entry points:
    tide_plan_create(shapes, N, M, L) -> plan handle
    tide_rs_reduce(plan, grads, shards, stream=None)
    tide_ag_place(plan, shards, params, elem_bytes, stream=None)
    tide_plan_destroy(plan)
plus the geometry/work-list queries and the ``TidePlan`` owner object.
"""

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
# TIDE_LIBRARY=checked loads the store-checked build (tests only).
LIB_PATH = os.path.join(HERE, "libtide_checked.so" if os.environ.get("TIDE_LIBRARY") == "checked" else "libtide.so")

TIDE_OK = 0
STATUS_NAMES = {
    0: "TIDE_OK", 1: "TIDE_ERR_INVALID_ARG", 2: "TIDE_ERR_ALIGNMENT", 3: "TIDE_ERR_OVERFLOW",
    4: "TIDE_ERR_OUT_OF_MEMORY", 5: "TIDE_ERR_CUDA", 6: "TIDE_ERR_UNIMPLEMENTED",
    7: "TIDE_ERR_DEVICE_MISMATCH", 8: "TIDE_ERR_TIMEOUT",
}
TIDE_OPT_RS_KERNEL = 1
TIDE_OPT_WAIT_LIMIT_NS = 2
TIDE_OPT_TEST_DROP_TILE = 3
TIDE_OPT_RS_AVERAGE = 4
TIDE_OPT_RS_ACCUMULATE = 5
TIDE_OPT_AG_UNPADDED = 6
TIDE_OPT_SUM_ORDER = 7
TIDE_OPT_CHECK_OVERLAP = 8
TIDE_OPT_RD_EXCHANGE = 9
TIDE_OPT_AG_TRANSPORT = 10
TIDE_AG_SM = 0
TIDE_AG_COPY_ENGINES = 1
TIDE_AG_BULK = 2
TIDE_SUM_LANDING = 0
TIDE_SUM_RELATIVE = 1
ITEM_FIELDS = ("kind", "p", "r", "src_off", "dst_off", "n")


class TideError(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class GroupDesc(ctypes.Structure):
    _fields_ = [("P", ctypes.c_int32), ("ndim", ctypes.POINTER(ctypes.c_int32)),
                ("dims", ctypes.POINTER(ctypes.c_int64)), ("N", ctypes.c_int32),
                ("M", ctypes.c_int32), ("L", ctypes.c_int32)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise TideError(-1, f"{LIB_PATH} is missing: build it with "
                            "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    sig = {
        "tide_plan_create": (i32, [ctypes.POINTER(GroupDesc), ctypes.POINTER(vp)]),
        "tide_plan_destroy": (None, [vp]),
        "tide_plan_shard_elems": (i64, [vp]),
        "tide_plan_param_geometry": (i32, [vp, i32] + [ctypes.POINTER(i64)] * 4),
        "tide_plan_num_items": (i64, [vp, i32]),
        "tide_plan_level2_order": (i32, [vp, i32, i32, ctypes.POINTER(i32)]),
        "tide_plan_get_items": (i32, [vp, i32, ctypes.POINTER(i64), i64]),
        "tide_rs_reduce": (i32, [vp, ctypes.POINTER(vp), ctypes.POINTER(vp), vp]),
        "tide_ag_place": (i32, [vp, ctypes.POINTER(vp), ctypes.POINTER(vp), i32, vp]),
        "tide_rs_reduce_noalloc": (i32, [vp, ctypes.POINTER(vp), ctypes.POINTER(vp), vp]),
        "tide_plan_set_option": (i32, [vp, i32, i64]),
        "tide_plan_check": (i32, [vp]),
        "tide_plan_last_launches": (i32, [vp]),
        "tide_debug_bounds_violations": (i64, [i32]),
        "tide_debug_bounds_selftest": (i32, []),
        "tide_slot_pack": (i32, [vp, ctypes.POINTER(vp), ctypes.POINTER(vp), vp]),
        "tide_rs_reduce_slots": (i32, [vp, ctypes.POINTER(vp), ctypes.POINTER(vp), vp]),
        "tide_plan_inbox_elems": (i64, [vp]),
        "tide_rs_staged": (i32, [vp, ctypes.POINTER(vp), ctypes.POINTER(vp), vp, i32, i32, vp]),
        "tide_rd_rounds": (i32, [i32]),
        "tide_rd_send_count": (i32, [i32, i32]),
        "tide_ag_rd_exchange": (i32, [vp, ctypes.POINTER(vp), i32, vp]),
        "tide_ag_stage_place": (i32, [vp, vp, i32, i32, ctypes.POINTER(vp), i32, vp]),
        "tide_ag_stage_init": (i32, [vp, ctypes.POINTER(vp), ctypes.POINTER(vp), i32, vp]),
        "tide_ag_rd_exchange_rails": (i32, [vp, ctypes.POINTER(vp), i32, vp]),
        "tide_status_string": (ctypes.c_char_p, [i32]),
        "tide_last_error": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()


def _check(status):
    if status != TIDE_OK:
        raise TideError(status, _lib.tide_last_error().decode() or
                        _lib.tide_status_string(status).decode())


def _ptr(x):
    """Device address of a tensor, or an int address, or None -> NULL."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ptr_array(items):
    if isinstance(items, PointerArray):
        return items.arr
    arr = (ctypes.c_void_p * len(items))()
    for i, x in enumerate(items):
        arr[i] = _ptr(x)
    return arr


class PointerArray:
    """A host array of device addresses, built once and passed to many calls.

    Building the C array from thousands of tensors costs milliseconds of
    Python time per call (12,336 gradient pointers for a 257-parameter group
    over 48 ranks); callers that reuse the same buffers build it once here.
    The tensors must stay alive and in place while the array is in use.
    """

    def __init__(self, items):
        self.arr = _ptr_array(list(items))
        self.n = len(self.arr)

    def __len__(self):
        return self.n


def pointer_array(items):
    return PointerArray(items)


def tide_plan_create(shapes, N, M, L):
    """Plan for a group of parameters with the given shapes (dim 0 first)."""
    shapes = [tuple(int(d) for d in s) for s in shapes]
    ndim = (ctypes.c_int32 * max(1, len(shapes)))(*[len(s) for s in shapes])
    flat = [d for s in shapes for d in s]
    dims = (ctypes.c_int64 * max(1, len(flat)))(*flat)
    desc = GroupDesc(len(shapes), ndim, dims, N, M, L)
    handle = ctypes.c_void_p()
    _check(_lib.tide_plan_create(ctypes.byref(desc), ctypes.byref(handle)))
    return handle.value


def tide_plan_destroy(plan):
    _lib.tide_plan_destroy(plan)


def tide_slot_pack(plan, grads, slots, stream=None):
    """Slot-Reuse: copy every rank's bf16 gradients into its all-gather slot."""
    _check(_lib.tide_slot_pack(plan, _ptr_array(grads), _ptr_array(slots), _stream(stream)))


def tide_rs_reduce_slots(plan, slots, shards, stream=None):
    """tide_rs_reduce reading every rank's gradients from its packed slot."""
    _check(_lib.tide_rs_reduce_slots(plan, _ptr_array(slots), _ptr_array(shards), _stream(stream)))


def tide_plan_inbox_elems(plan):
    return int(_lib.tide_plan_inbox_elems(plan))


def tide_rs_staged(plan, grads, shards, inbox, sum_ctas_per_rank=0, landing_ctas_per_rank=0, stream=None):
    """Two-stage reduce-scatter through an explicit inbox (same bits as tide_rs_reduce)."""
    _check(_lib.tide_rs_staged(plan, _ptr_array(grads), _ptr_array(shards), _ptr(inbox), sum_ctas_per_rank,
                               landing_ctas_per_rank, _stream(stream)))


def tide_rd_rounds(M):
    return int(_lib.tide_rd_rounds(M))


def tide_rd_send_count(M, d):
    return int(_lib.tide_rd_send_count(M, d))


def tide_ag_rd_exchange(plan, stages, elem_bytes, stream=None):
    """stages: M device buffers of M*S elements (slot 0 = the node's own shard)."""
    _check(_lib.tide_ag_rd_exchange(plan, _ptr_array(stages), elem_bytes, _stream(stream)))


def tide_ag_stage_place(plan, stage, node, rail, params, elem_bytes, stream=None):
    _check(_lib.tide_ag_stage_place(plan, _ptr(stage), node, rail, _ptr_array(params), elem_bytes,
                                    _stream(stream)))


def tide_ag_stage_init(plan, shards, stages, elem_bytes, stream=None):
    """shards: N device buffers; stages: L*M stage buffers (rail l's node n at l*M + n)."""
    _check(_lib.tide_ag_stage_init(plan, _ptr_array(shards), _ptr_array(stages), elem_bytes, _stream(stream)))


def tide_ag_rd_exchange_rails(plan, stages, elem_bytes, stream=None):
    """stages: L*M device buffers of M*S elements, rail l's node n at l*M + n."""
    _check(_lib.tide_ag_rd_exchange_rails(plan, _ptr_array(stages), elem_bytes, _stream(stream)))


def stage_shard_pointers(stages, node, M, L, S, elem_bytes):
    """Addresses that make tide_ag_place place node `node`'s pieces of every
    rail from the stage buffers (rail l's node n at l*M + n): rank r's shard
    is slot (r // L - node) mod M of stages[(r % L) * M + node]."""
    base = [_ptr(x) for x in stages]
    return [base[(r % L) * M + node] + ((r // L - node) % M) * S * elem_bytes for r in range(M * L)]


def tide_plan_set_option(plan, option, value):
    _check(_lib.tide_plan_set_option(plan, option, value))


def tide_plan_check(plan):
    """Synchronise and raise TideError(TIDE_ERR_TIMEOUT) if a kernel gave up a wait."""
    _check(_lib.tide_plan_check(plan))


def tide_plan_shard_elems(plan):
    return int(_lib.tide_plan_shard_elems(plan))


def tide_plan_param_geometry(plan, p):
    """(R_p, Rp, Kp, op) of parameter p."""
    out = [ctypes.c_int64() for _ in range(4)]
    _check(_lib.tide_plan_param_geometry(plan, p, *[ctypes.byref(o) for o in out]))
    return tuple(int(o.value) for o in out)


def tide_plan_level2_order(plan, n_dest, s, M):
    """Source nodes of slice s of destination node n_dest, in summation order."""
    out = (ctypes.c_int32 * M)()
    _check(_lib.tide_plan_level2_order(plan, n_dest, s, out))
    return list(out)


def tide_debug_bounds_violations(reset=False):
    """Stores the checked build skipped since the last reset (-1: normal build)."""
    return int(_lib.tide_debug_bounds_violations(1 if reset else 0))


def tide_debug_bounds_selftest():
    """One deliberate out-of-range check with no memory access (positive control)."""
    _check(_lib.tide_debug_bounds_selftest())


def tide_plan_items(plan, which):
    """Work list as a list of dicts (which=0: reduce-scatter, 1: all-gather,
    2 / 3: the all-gather split for bulk copies: aligned middles / the rest)."""
    n = int(_lib.tide_plan_num_items(plan, which))
    if n < 0:
        raise TideError(1, "bad plan or list selector")
    buf = (ctypes.c_int64 * max(1, 6 * n))()
    _check(_lib.tide_plan_get_items(plan, which, buf, n))
    return [dict(zip(ITEM_FIELDS, buf[6 * i:6 * i + 6])) for i in range(n)]


def tide_rs_reduce(plan, grads, shards, stream=None):
    """grads: N*P tensors/addresses (entry r*P + p), shards: N fp32 tensors/addresses."""
    _check(_lib.tide_rs_reduce(plan, _ptr_array(grads), _ptr_array(shards), _stream(stream)))


def tide_rs_reduce_noalloc(plan, grads, shards, stream=None):
    """tide_rs_reduce without any device allocation (fixed static scratch)."""
    _check(_lib.tide_rs_reduce_noalloc(plan, _ptr_array(grads), _ptr_array(shards), _stream(stream)))


def tide_ag_place(plan, shards, params, elem_bytes, stream=None):
    """shards: N tensors/addresses of S elements, params: P tensors/addresses."""
    _check(_lib.tide_ag_place(plan, _ptr_array(shards), _ptr_array(params), elem_bytes, _stream(stream)))


class TidePlan:
    """Owns a plan handle; geometry is read back from the library."""

    def __init__(self, shapes, N, M, L):
        self.shapes = [tuple(s) for s in shapes]
        self.N, self.M, self.L = N, M, L
        self.handle = tide_plan_create(self.shapes, N, M, L)
        self.S = tide_plan_shard_elems(self.handle)
        self.P = len(self.shapes)
        geo = [tide_plan_param_geometry(self.handle, p) for p in range(self.P)]
        self.rows = [g[0] for g in geo]
        self.Rp = [g[1] for g in geo]
        self.Kp = [g[2] for g in geo]
        self.o = [g[3] for g in geo]
        self.e = [g[1] * g[2] for g in geo]

    def rs_reduce(self, grads, shards, stream=None):
        tide_rs_reduce(self.handle, grads, shards, stream)

    def ag_place(self, shards, params, elem_bytes, stream=None):
        tide_ag_place(self.handle, shards, params, elem_bytes, stream)

    def items(self, which):
        return tide_plan_items(self.handle, which)

    def set_option(self, option, value):
        tide_plan_set_option(self.handle, option, value)

    def check(self):
        tide_plan_check(self.handle)

    def last_launches(self):
        """Kernels launched by the plan's most recent compute call."""
        return int(_lib.tide_plan_last_launches(self.handle))

    def level2_order(self, n_dest, s):
        return tide_plan_level2_order(self.handle, n_dest, s, self.M)

    def close(self):
        if self.handle:
            tide_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
