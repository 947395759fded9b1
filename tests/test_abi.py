"""The C-ABI library, checked without a GPU.

librssm.so must load and export every function declared in include/rssm.h.
The host-side validation and the buffer layouts are checked here too (no
compute call runs).
"""
import ctypes
import os
import re

import pytest

from hybrid_model_ssm_gb300 import LayerShape, RssmError, read_copy_layout, ring_offsets, workspace_size
from hybrid_model_ssm_gb300 import build as build_mod
from hybrid_model_ssm_gb300.rssm import RSSM_EINVAL, RSSM_EUNSUPPORTED, SIGNATURES

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rssm.h")


@pytest.fixture(scope="module")
def lib():
    path = build_mod.build()  # nvcc cross-compiles without a GPU; a no-op when up to date
    return ctypes.CDLL(path)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rssm_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_function_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), f"{n} declared in rssm.h but not exported"


def test_binding_covers_the_header():
    assert set(declared_functions()) == set(SIGNATURES)


def test_workspace_layout_of_the_layer_workload(lib):
    s = LayerShape(B=256, H=128, P=64, N=128, G=8, L=16)
    ring, ptrs, copy = workspace_size(s)
    v_off, k_off = ring_offsets(s)
    R, Rp = 16, 16
    assert v_off == 256 * 128 * Rp * 4
    assert k_off == v_off + 256 * 128 * R * 64 * 2
    assert ring == k_off + 256 * 8 * R * 128 * 2
    assert v_off % 256 == 0 and k_off % 256 == 0
    assert ptrs == 5 * 1024 + 512  # start, count, ticket, error word (256 B), epoch, flush list, its length
    assert copy == 0


def test_read_copy_layouts(lib):
    e4 = LayerShape(B=2, H=4, P=64, N=128, G=2, L=16, read_fmt="e4m3")
    stride, bsc, rsc = read_copy_layout(e4)
    assert (stride, rsc) == (64 * 128 + 4 * 64, 64 * 128)
    e2 = LayerShape(B=2, H=4, P=64, N=128, G=2, L=16, read_fmt="e2m1")
    stride, bsc, rsc = read_copy_layout(e2)
    assert bsc == 64 * 64 and rsc == bsc + 64 * 8 and stride == rsc + 256
    assert workspace_size(e2)[2] == 2 * 4 * stride
    with pytest.raises(RssmError):
        read_copy_layout(LayerShape(B=2, H=4, P=64, N=128, G=2, L=16))


@pytest.mark.parametrize("kw,status", [
    (dict(H=3, G=2), RSSM_EINVAL),
    (dict(N=48), RSSM_EUNSUPPORTED),
    (dict(N=256), RSSM_EUNSUPPORTED),
    (dict(P=12), RSSM_EUNSUPPORTED),
    (dict(B=0), RSSM_EINVAL),
    (dict(L=30, T_max=4), RSSM_EUNSUPPORTED),
    (dict(T_max=9), RSSM_EUNSUPPORTED),
    (dict(N=32, read_fmt="e2m1"), RSSM_EUNSUPPORTED),
    (dict(P=256, N=128), RSSM_EUNSUPPORTED),
    # two f32 tiles of 128 x 128, two record slots and the group areas overflow shared memory
    (dict(P=128, N=128, L=30, in_dtype="f32"), RSSM_EUNSUPPORTED),
    (dict(P=128, N=128, L=27, T_max=4, in_dtype="f32"), RSSM_EUNSUPPORTED),
    (dict(P=128, N=128, L=29, in_dtype="f32", recurrence="delta"), RSSM_EUNSUPPORTED),
])
def test_invalid_configurations_are_rejected(lib, kw, status):
    base = dict(B=2, H=4, P=16, N=64, G=2, L=4, T_max=1)
    base.update(kw)
    with pytest.raises(RssmError) as ei:
        workspace_size(LayerShape(**base))
    assert ei.value.status == status


@pytest.mark.parametrize("kw", [
    dict(P=128, N=128, L=29, in_dtype="f32"),
    dict(P=128, N=128, L=26, T_max=4, in_dtype="f32"),
    dict(P=128, N=128, L=28, in_dtype="f32", recurrence="delta"),
    dict(P=128, N=128, L=32),
    dict(P=128, N=128, L=25, T_max=8),
    dict(P=128, N=128, L=32, recurrence="delta"),
    dict(P=120, N=128, L=32, in_dtype="f32"),
])
def test_largest_placeable_configurations_are_accepted(lib, kw):
    """The edge of the shared-memory plan: each of these still fits one CTA."""
    base = dict(B=2, H=4, G=2, T_max=1)
    base.update(kw)
    ring, ptrs, _ = workspace_size(LayerShape(**base))
    assert ring > 0 and ptrs > 0


def test_launch_plans_keep_the_ring_rule_over_the_size_grid(lib):
    """Host planner over a grid of sizes, formats and recurrences (no CUDA call).

    Every plan fits 227 KiB and keeps each shared-memory ring's length a multiple
    of the consumers that take its entries in turn (stages: the dot groups;
    slots: max(2, dot groups)), the rule that keeps an mbarrier parity wait from
    matching the previous phase. A configuration is accepted by the sizing call
    exactly when all of its launches can be planned."""
    from hybrid_model_ssm_gb300 import launch_plan
    smem_max = 227 * 1024
    windows = [(1, 1), (2, 1), (4, 1), (16, 1), (29, 1), (32, 1), (2, 2), (4, 4), (16, 4), (27, 4), (8, 8), (25, 8)]
    planned = refused = 0
    for N in (16, 32, 64, 128):
        for P in (8, 24, 64, 120, 128):
            for L, T in windows:
                for dt in ("f32", "bf16"):
                    for rf, ck, rec in (("none", "f32", "outer"), ("e4m3", "f32", "outer"), ("e2m1", "f32", "outer"),
                                        ("none", "f16_sr", "outer"), ("none", "f32", "delta")):
                        shape = LayerShape(B=3, H=4, P=P, N=N, G=2, L=L, T_max=T, in_dtype=dt, read_fmt=rf, ckpt=ck,
                                           recurrence=rec)
                        kinds = ["flush", "decode"] + (["verify"] if T > 1 else [])
                        plans = {}
                        for kind in kinds:
                            try:
                                plans[kind] = launch_plan(shape, kind)
                            except RssmError:
                                pass
                        try:
                            workspace_size(shape)
                            accepted = True
                        except RssmError:
                            accepted = False
                        assert accepted == (len(plans) == len(kinds)), (shape, sorted(plans))
                        if not accepted:
                            refused += 1
                            continue
                        planned += 1
                        ck_es = 2 if ck != "f32" else 4
                        for kind, plan in plans.items():
                            assert 0 < plan["smem_bytes"] <= smem_max
                            for i, lay in enumerate(plan["layouts"]):
                                d = lay["dgroups"]
                                assert d in (1, 2, 4, 8) and lay["stages"] >= 2
                                assert lay["stages"] % d == 0 and lay["slots"] % max(2, d) == 0, (shape, kind, lay)
                                assert lay["stage_bytes"] % 128 == 0 and lay["slot_bytes"] % 128 == 0
                                assert lay["stages"] * lay["stage_bytes"] + lay["slots"] * lay["slot_bytes"] \
                                    <= plan["smem_bytes"]
                                if i == 0:  # the general layout holds a whole checkpoint tile
                                    assert lay["stage_bytes"] >= P * N * ck_es
    assert planned > 500 and refused > 100


def test_warp_per_head_plans_over_the_size_grid(lib):
    """Host planner of the warp-per-head non-flush step (no CUDA call): for every accepted
    read-copy or FP16 configuration of the grid, each warp's two tile stages hold the head's
    tile (the copy's head stride, or P x N binary16 values) and the ring's decays at the next
    16-byte boundary, its value stage holds the L - 1 value rows a non-flush step can read,
    and the CTA takes as many warps as 227 KiB allow, up to 16. Other layers have no such plan."""
    from hybrid_model_ssm_gb300 import launch_plan
    smem_max, cta_bytes, bar_bytes = 227 * 1024, 128, 32
    planned = 0
    for N in (64, 128):
        for P in (8, 24, 64, 120, 128):
            for L, T in ((1, 1), (2, 1), (4, 1), (16, 1), (32, 1), (16, 4), (25, 8)):
                for dt, es in (("f32", 4), ("bf16", 2)):
                    for fmt in ("e4m3", "e2m1", "f16_sr", "f16_rn"):
                        kw = dict(ckpt=fmt) if fmt.startswith("f16") else dict(read_fmt=fmt)
                        shape = LayerShape(B=3, H=4, P=P, N=N, G=2, L=L, T_max=T, in_dtype=dt, **kw)
                        try:
                            workspace_size(shape)
                        except RssmError:
                            continue
                        plan = launch_plan(shape, "warp_per_head")
                        (lay,) = plan["layouts"]
                        tile = P * N * 2 if fmt.startswith("f16") else read_copy_layout(shape)[0]
                        Rp = (L + T - 1 + 3) // 4 * 4
                        warps = lay["dgroups"]
                        assert lay["stages"] == 2 and lay["slots"] == 1
                        assert lay["stage_bytes"] % 128 == 0 and lay["slot_bytes"] % 128 == 0
                        assert lay["stage_bytes"] >= (tile + 15) // 16 * 16 + 4 * Rp
                        assert lay["slot_bytes"] >= max(L - 1, 1) * P * es
                        per_warp = bar_bytes + (P * 4 + 127) // 128 * 128 + 2 * lay["stage_bytes"] + lay["slot_bytes"]
                        assert plan["smem_bytes"] == cta_bytes + warps * per_warp <= smem_max, (shape, plan)
                        assert 1 <= warps <= 16
                        assert warps == 16 or cta_bytes + (warps + 1) * per_warp > smem_max, (shape, plan)
                        planned += 1
    assert planned > 200
    # the read-copy decode workload (B=256 H=128 P=64 N=128 G=8 L=16, bf16 inputs):
    # 12 warps per CTA with an E4M3 copy, 16 with an E2M1 copy
    for fmt, warps in (("e4m3", 12), ("e2m1", 16)):
        shape = LayerShape(B=256, H=128, P=64, N=128, G=8, L=16, in_dtype="bf16", read_fmt=fmt)
        assert launch_plan(shape, "warp_per_head")["layouts"][0]["dgroups"] == warps
    for kw in (dict(), dict(recurrence="delta")):
        with pytest.raises(RssmError, match="EUNSUPPORTED"):
            launch_plan(LayerShape(B=2, H=4, P=64, N=128, G=2, L=16, **kw), "warp_per_head")


def test_null_config_and_handle(lib):
    lib.rssm_workspace_size.restype = ctypes.c_int
    assert lib.rssm_workspace_size(None, None, None, None) == RSSM_EINVAL
    lib.rssm_decode_step.restype = ctypes.c_int
    assert lib.rssm_decode_step(None, None, None, None, None, None, None) == RSSM_EINVAL
    lib.rssm_last_error.restype = ctypes.c_char_p
    assert b"NULL" in lib.rssm_last_error()
    assert lib.rssm_destroy(None) == 0


def test_config_struct_matches_the_header(tmp_path):
    """ctypes' Config against the C compiler's layout of rssm_config."""
    from hybrid_model_ssm_gb300.rssm import Config
    src = tmp_path / "layout.c"
    fields = [f for f, _ in Config._fields_]
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "rssm.h"\nint main(void) {\n'
                   '  printf("%zu", sizeof(rssm_config));\n'
                   + "".join(f'  printf(" %zu", offsetof(rssm_config, {f}));\n' for f in fields)
                   + "  return 0;\n}\n")
    exe = tmp_path / "layout"
    import subprocess
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    assert got[0] == ctypes.sizeof(Config)
    assert got[1:] == [getattr(Config, f).offset for f in fields]


def test_launch_plan_struct_matches_the_header(tmp_path):
    """ctypes' LaunchPlanInfo against the C compiler's layout of rssm_launch_plan_info."""
    import subprocess

    from hybrid_model_ssm_gb300.rssm import LaunchPlanInfo
    fields = [f for f, _ in LaunchPlanInfo._fields_]
    src = tmp_path / "plan_layout.c"
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "rssm.h"\nint main(void) {\n'
                   '  printf("%zu", sizeof(rssm_launch_plan_info));\n'
                   + "".join(f'  printf(" %zu", offsetof(rssm_launch_plan_info, {f}));\n' for f in fields)
                   + "  return 0;\n}\n")
    exe = tmp_path / "plan_layout"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    assert got[0] == ctypes.sizeof(LaunchPlanInfo)
    assert got[1:] == [getattr(LaunchPlanInfo, f).offset for f in fields]


def test_delta_rule_ring_layout(lib):
    """Delta-rule layers keep fp32 pseudo-values [B,H,R,P] where V sits."""
    s = LayerShape(B=3, H=4, P=64, N=128, G=2, L=5, recurrence="delta")
    Rp, R = 8, 5
    up = lambda x: (x + 255) // 256 * 256  # noqa: E731
    v_off, k_off = ring_offsets(s)
    assert v_off == up(3 * 4 * Rp * 4)
    assert k_off == up(v_off + 3 * 4 * R * 64 * 4)
    assert workspace_size(s)[0] == up(k_off + 3 * 2 * R * 128 * 2)


@pytest.mark.parametrize("kw,status", [
    (dict(N=32), RSSM_EUNSUPPORTED),
    (dict(T_max=5), RSSM_EUNSUPPORTED),  # delta-rule verify takes at most 4 drafts
    (dict(read_fmt="e4m3"), RSSM_EUNSUPPORTED),
    (dict(ckpt="f16_sr"), RSSM_EUNSUPPORTED),
])
def test_delta_rule_configurations_are_limited(lib, kw, status):
    base = dict(B=2, H=4, P=16, N=64, G=2, L=4, T_max=1, recurrence="delta")
    base.update(kw)
    with pytest.raises(RssmError) as ei:
        workspace_size(LayerShape(**base))
    assert ei.value.status == status


def test_unknown_recurrence_is_rejected(lib):
    from hybrid_model_ssm_gb300.rssm import Config
    cfg = LayerShape(B=2, H=4, P=16, N=64, G=2, L=4).config()
    cfg.recurrence = 7
    r, p, q = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    lib.rssm_workspace_size.restype = ctypes.c_int
    assert lib.rssm_workspace_size(ctypes.byref(cfg), ctypes.byref(r), ctypes.byref(p), ctypes.byref(q)) == RSSM_EINVAL
    assert isinstance(cfg, Config)


@pytest.mark.parametrize("compiler,std", [("gcc", "-std=c99"), ("g++", "-std=c++17")])
def test_header_compiles_cleanly(tmp_path, compiler, std):
    """include/rssm.h is plain C: it compiles as C99 and as C++17 with every warning an error."""
    import subprocess
    src = tmp_path / "use_header.c"
    src.write_text('#include "rssm.h"\nint main(void) { return (int)(sizeof(rssm_config) + sizeof(rssm_launch_plan_info)) == 0; }\n')
    lang = ["-x", "c++"] if compiler == "g++" else []
    subprocess.run([compiler, std, "-Wall", "-Wextra", "-pedantic", "-Werror", *lang, "-I",
                    os.path.join(ROOT, "include"), str(src), "-o", str(tmp_path / "use_header")], check=True)
