"""TIDE layout-aware FSDP2 collectives, single-GPU hot path for GB300 (sm_103a).

``tide_rs_reduce`` and ``tide_ag_place`` run in hand-written CUDA kernels in
``libtide.so`` (C ABI: include/tide.h); this package only binds them.
"""

from .tide import (  # noqa: F401
    LIB_PATH, PointerArray, TideError, TidePlan, pointer_array,
    tide_plan_create, tide_plan_destroy, tide_plan_items, tide_plan_level2_order, tide_plan_param_geometry,
    tide_plan_shard_elems, tide_plan_set_option, tide_plan_check, tide_plan_inbox_elems,
    tide_rs_reduce, tide_rs_reduce_noalloc, tide_rs_staged, tide_rs_reduce_slots, tide_slot_pack,
    tide_ag_place, tide_rd_rounds, tide_rd_send_count, tide_ag_rd_exchange, tide_ag_stage_place,
    tide_ag_stage_init, tide_ag_rd_exchange_rails, stage_shard_pointers,
    tide_debug_bounds_violations, tide_debug_bounds_selftest,
    TIDE_OPT_RS_KERNEL, TIDE_OPT_WAIT_LIMIT_NS, TIDE_OPT_TEST_DROP_TILE, TIDE_OPT_RS_AVERAGE,
    TIDE_OPT_RS_ACCUMULATE, TIDE_OPT_AG_UNPADDED, TIDE_OPT_SUM_ORDER, TIDE_OPT_CHECK_OVERLAP,
    TIDE_OPT_RD_EXCHANGE, TIDE_OPT_AG_TRANSPORT,
    TIDE_SUM_LANDING, TIDE_SUM_RELATIVE, TIDE_AG_SM, TIDE_AG_COPY_ENGINES, TIDE_AG_BULK,
)
