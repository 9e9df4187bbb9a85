"""The C ABI without a GPU: the library builds, loads, exports every symbol
include/moe.h declares, and its host-side validation and workspace query
(which touch no CUDA call) behave as documented."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from combine_route_scan_gb300 import build
    build.build()
    from combine_route_scan_gb300 import moe
    return moe


def declared_functions():
    with open(os.path.join(ROOT, "include", "moe.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:moe_status_t|const char\*)\s+(moe_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_abi():
    assert declared_functions() == sorted(
        ["moe_get_workspace_size", "moe_workspace_init", "moe_dispatch", "moe_combine",
         "moe_dispatch_ffn_combine", "moe_combine_noalloc", "moe_get_device_status", "moe_status_string"])


def test_library_exports_every_declared_symbol(lib):
    L = lib.lib()
    for name in declared_functions():
        assert hasattr(L, name), name
    assert set(lib.EXPORTS) == set(declared_functions())


def test_config_struct_layout_matches_header(lib):
    # 17 int32/int64 fields plus a pointer: offsets follow C layout rules
    assert ctypes.sizeof(lib.MoeConfig) == 104
    assert lib.MoeConfig.bulk_min_bytes.offset == 48
    assert lib.MoeConfig.prof_events.offset == 72
    assert lib.MoeConfig.seg_ready.offset == 80
    assert lib.MoeConfig.seg_ready_ticket.offset == 88
    assert lib.MoeConfig.performance_info.offset == 96


def test_workspace_query_and_capacity(lib):
    import torch
    cfg = lib.config(16, 256, 7168, 8, 256, torch.bfloat16, zero_expert_num=4, copy_expert_num=4, mask_kind=2)
    n, A = lib.workspace_size(cfg)
    assert A == 256 * 16 * min(16, 8)
    assert n > 0 and n % 256 == 0
    cfg2 = lib.config(16, 256, 7168, 8, 256, torch.bfloat16, combine_mode=lib.COMBINE_TWO_PHASE)
    n2, _ = lib.workspace_size(cfg2)
    # the two-phase window holds one row per pick
    assert n2 - n >= 16 * 256 * 8 * 7168 * 2
    cfg3 = lib.config(2, 8, 16, 2, 4, torch.int32)
    assert lib.workspace_size(cfg3)[1] == 8 * 2 * 2


@pytest.mark.parametrize("field,value,code", [
    ("ep_world_size", 1, "INVALID_ARG"),
    ("ep_world_size", 769, "INVALID_ARG"),
    ("moe_expert_num", 0, "INVALID_ARG"),
    ("moe_expert_num", 1025, "INVALID_ARG"),
    ("moe_expert_num", 63, "INVALID_ARG"),
    ("topk", 0, "INVALID_ARG"),
    ("topk", 33, "INVALID_ARG"),
    ("h", 0, "INVALID_ARG"),
    ("bs", -1, "INVALID_ARG"),
    ("const_expert_num", 1, "UNSUPPORTED"),
    ("quant_mode", 1, "INVALID_ARG"),      # static quantisation needs a scales input
    ("quant_mode", 3, "INVALID_ARG"),      # per-group needs an FP8 expand_dtype
    ("quant_mode", 5, "UNSUPPORTED"),
    ("expand_dtype", 1, "INVALID_ARG"),    # quantised types only with quant_mode 3 / 4
    ("scales_kind", 3, "INVALID_ARG"),
    ("mask_kind", 3, "INVALID_ARG"),
    ("x_dtype", 7, "INVALID_ARG"),
    ("plane_policy", 3, "INVALID_ARG"),
    ("combine_mode", 3, "INVALID_ARG"),
    ("wait_timeout_us", 0, "INVALID_ARG"),
    ("bulk_min_bytes", -1, "INVALID_ARG"),
])
def test_host_validation(lib, field, value, code):
    import torch
    cfg = lib.config(8, 32, 7168, 8, 64, torch.float16)
    setattr(cfg, field, value)
    with pytest.raises(lib.MoeError) as ei:
        lib.workspace_size(cfg)
    assert ei.value.name == code


def test_quant_with_int32_is_rejected(lib):
    import torch
    cfg = lib.config(8, 32, 7168, 8, 64, torch.int32, quant_mode=2)
    with pytest.raises(lib.MoeError) as ei:
        lib.workspace_size(cfg)
    assert ei.value.name == "UNSUPPORTED"


def test_status_strings(lib):
    for code in range(11):
        assert lib.status_string(code) != "unknown status"


def test_binding_refuses_cpu_tensors(lib):
    import torch
    cfg = lib.config(2, 8, 16, 2, 4, torch.int32)
    x = torch.zeros(2, 8, 16, dtype=torch.int32)
    with pytest.raises(ValueError):
        lib.dispatch(cfg, x, x, None, None, x, None, x, x, ws=x)


def test_quant_rules_agree_with_oracle(lib):
    """The library's host validation of quant_mode / expand_dtype / scales_kind
    gives the same verdict as the oracle's configuration rules, over every
    combination (and an odd h, which FP4 rows cannot pack)."""
    import itertools
    import torch
    import workloads as WL
    from oracle import oracle as O
    names = {v: k for k, v in O.Y_KIND.items() if k != "int8"}
    code = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED"}
    for xdt, q, y, k, h in itertools.product((torch.bfloat16, torch.int32), range(6), range(4), range(4), (64, 63)):
        cfg = lib.config(4, 8, h, 2, 8, xdt, quant_mode=q, expand_dtype=y, scales_kind=k)
        try:
            lib.workspace_size(cfg)
            got = "OK"
        except lib.MoeError as e:
            got = e.name
        wl = WL.Workload("r", 4, 8, h, 2, 8, WL.X_BF16 if xdt == torch.bfloat16 else WL.X_INT32, quant_mode=q,
                         y_dtype=names[y], scales_kind=k)
        cfgo = O.make_cfg(wl)
        cfgo.y_kind, cfgo.scales_kind = y, k  # also when quant_mode is 0
        want = code[int(O.lib().orc_check_cfg(ctypes.byref(cfgo)))]
        assert got == want, (xdt, q, y, k, h, got, want)
