"""CPU-only checks of the C ABI library: it loads without a GPU, exports every symbol the
header declares, and its host-side validation and workspace layout behave as documented
(none of these calls touches the device)."""
import ctypes
import math
import os
import re
import subprocess

import pytest

import grouped_gemm_device_gb300 as g
from grouped_gemm_device_gb300 import build as gbuild
from grouped_gemm_device_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return g.load()


def header_functions():
    src = open(os.path.join(ROOT, "include", "moegmm.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", src, re.M)
    return sorted(set(n for n in names if n not in ("if", "defined")))


def test_exports_every_declared_symbol(lib):
    declared = header_functions()
    assert set(declared) >= {"moe_route_permute", "moe_grouped_mlp_fwd", "moe_grouped_mlp_bwd",
                             "mxfp8_quantize", "moe_pack_fc1_weight", "moe_workspace_size"}
    out = subprocess.run(["nm", "-D", "--defined-only", g.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\b[TW] (\w+)$", out, re.M))
    missing = [n for n in declared if n not in exported]
    assert not missing, missing
    assert set(g.EXPORTS) <= exported


def test_desc_struct_layout_matches_header(lib, tmp_path):
    # the binding's ctypes structures against the C compiler's view of the header
    src = tmp_path / "sz.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "moegmm.h"\n'
                   'int main(void) { printf("%zu %zu %zu\\n", sizeof(moe_layer_desc_t), '
                   'sizeof(moe_ws_layout_t), offsetof(moe_layer_desc_t, reuse_weights));'
                   ' return 0; }\n')
    exe = tmp_path / "sz"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True)
    desc, ws, reuse = map(int, subprocess.run([str(exe)], capture_output=True, text=True,
                                              check=True).stdout.split())
    assert ctypes.sizeof(g.LayerDesc) == desc == 20 * 4
    assert g.LayerDesc.reuse_weights.offset == reuse
    assert ctypes.sizeof(g.WsLayout) == ws == 19 * 8


def _desc(**kw):
    base = dict(E=8, k=2, H=256, F=512, T_max=1000)
    base.update(kw)
    return g.make_desc(**base)


def test_workspace_layout_is_consistent(lib):
    d = _desc()
    L = g.moe_workspace_layout(d)
    assert L.total == g.moe_workspace_size(d)
    R = 1000 * 2 + 8 * 31
    assert L.R_cap == R
    fields = ["err", "offsets", "row_of", "src_of", "row_prob", "x_perm", "z", "a_s", "y_perm",
              "dy_perm", "dz", "dprob_part"]
    offs = [getattr(L, f) for f in fields]
    assert offs[0] == 0 and all(o % 256 == 0 for o in offs)
    assert offs == sorted(offs)
    assert L.z - L.x_perm >= R * 256 * 2
    assert L.a_s - L.z >= R * 1024 * 2
    assert L.dx_perm == L.y_perm
    assert L.total >= L.dprob_part + R * 2 * 4


@pytest.mark.parametrize("prec", [dict(), dict(precision="mxfp8", align=128),
                                  dict(precision="nvfp4", align=128)])
def test_recompute_keeps_no_z_in_the_workspace(lib, prec):
    keep, rc = _desc(**prec), _desc(recompute=True, **prec)
    Lk, Lr = g.moe_workspace_layout(keep), g.moe_workspace_layout(rc)
    assert Lk.z != 2 ** 64 - 1 and Lr.z == 2 ** 64 - 1  # SIZE_MAX: no saved FC1 output
    # the saved Z is R_cap x N1 bf16; the recomputing kernels' d_prob partials (narrower
    # tiles, more partials a row) take back at most 16 fp32 a row
    saved = Lk.R_cap * 1024 * 2
    assert Lk.total - Lr.total >= saved - Lk.R_cap * 16 * 4 - 4096


@pytest.mark.parametrize("kw,status", [
    (dict(E=0), 1), (dict(E=300), 1), (dict(k=0), 1), (dict(k=9, E=16), 1), (dict(k=5, E=4), 1),
    (dict(H=100), 2), (dict(F=96), 2), (dict(align=16), 2), (dict(ilv=48), 2),
    (dict(F=64 * 3, ilv=128), 2), (dict(sm_margin=-1), 1),
    (dict(precision="mxfp8"), 2), (dict(precision="mxfp8", align=128, ilv=128), 2),
    (dict(recompute=2), 1),
    (dict(extras=4), 1), (dict(extras=1, activation="srelu"), 2),
    (dict(extras=3, precision="mxfp8", align=128, activation="srelu"), 2),
    (dict(extras=1, recompute=1), 2),
    (dict(precision="nvfp4"), 2), (dict(precision="nvfp4", align=128, ilv=32), 2),
    (dict(precision="nvfp4", align=128, extras=1, activation="srelu"), 2),
])
def test_invalid_descriptions_rejected(lib, kw, status):
    d = _desc(**kw)
    assert lib.moe_workspace_size(ctypes.byref(d)) == 0
    with pytest.raises(g.MoeError) as ei:
        g.moe_workspace_layout(d)
    assert ei.value.status == status


def test_nvfp4_layout(lib):
    d = _desc(precision="nvfp4", align=128, rht_mask=0x1234)
    L = g.moe_workspace_layout(d)
    R, H, F, N1, E = L.R_cap, 256, 512, 1024, 8
    assert R % 128 == 0 and R >= 1000 * 2 + 8 * 127
    assert L.mx_base == 2 ** 64 - 1 and L.nv_amax != 2 ** 64 - 1
    assert L.a_s != 2 ** 64 - 1 and L.dz != 2 ** 64 - 1 and L.z != 2 ** 64 - 1
    assert L.nv_amax % 256 == 0 and L.nv_base >= L.nv_amax + 16 * 4
    # twelve operand copies at half a byte a value, each with its scales
    values = 2 * (R * H + R * F + R * H + R * N1) + 2 * (E * N1 * H + E * F * H)
    assert L.total - L.nv_base >= values // 2 + values // 16
    sd = g.moe_workspace_layout(_desc(precision="nvfp4", align=128, activation="srelu", ilv=0))
    assert sd.total < L.total


def test_nvfp4_entry_points_validate_on_the_host(lib):
    with pytest.raises(g.MoeError) as e:   # M not a multiple of 128
        g.nvfp4_quantize(256, 100, 64, 256, 256, 0, 0, 256, 256, None, None, 0)
    assert e.value.status == 2
    with pytest.raises(g.MoeError) as e:   # N not a multiple of 64
        g.nvfp4_quantize(256, 128, 96, 256, 256, 0, 0, 256, 256, None, None, 0)
    assert e.value.status == 2
    with pytest.raises(g.MoeError) as e:   # no copy requested
        g.nvfp4_quantize(256, 128, 64, 256, 256, 0, 0, None, None, None, None, 0)
    assert e.value.status == 1
    with pytest.raises(g.MoeError) as e:   # q_row not 32-byte aligned
        g.nvfp4_quantize(256, 128, 64, 256, 256, 0, 0, 272, 256, None, None, 0)
    assert e.value.status == 1
    with pytest.raises(g.MoeError) as e:   # transposed copy without its amax
        g.nvfp4_quantize(256, 128, 64, 256, None, 1, 0, None, None, 256, 256, 0)
    assert e.value.status == 1
    with pytest.raises(g.MoeError) as e:   # rotated amax needs whole 16-row blocks
        g.nvfp4_amax(256, 24, 64, 0, 256, 512, 0)
    assert e.value.status == 2
    with pytest.raises(g.MoeError) as e:
        g.nvfp4_amax(256, 16, 64, 0, None, None, 0)
    assert e.value.status == 1


def test_srelu_allows_any_ilv(lib):
    d = _desc(activation="srelu", ilv=0)
    L = g.moe_workspace_layout(d)
    assert L.a_s - L.z >= L.R_cap * 512 * 2


def test_calls_validate_before_touching_the_device(lib):
    d = _desc()
    n = g.moe_workspace_size(d)
    # T beyond capacity, NULL pointers, small or misaligned workspace: rejected on the host
    with pytest.raises(g.MoeError) as e:
        g.moe_route_permute(d, 1001, 16, 16, 16, 16, 16, 256, n, 0)
    assert e.value.status == 1
    with pytest.raises(g.MoeError) as e:
        g.moe_route_permute(d, 10, None, 16, 16, 16, 16, 256, n, 0)
    assert e.value.status == 1
    with pytest.raises(g.MoeError) as e:
        g.moe_grouped_mlp_fwd(d, 10, 256, 256, 256, 256, n - 1, 0)
    assert e.value.status == 3
    with pytest.raises(g.MoeError) as e:
        g.moe_grouped_mlp_fwd(d, 10, 256, 256, 256, 257, n, 0)
    assert e.value.status == 1
    with pytest.raises(g.MoeError) as e:
        g.moe_grouped_mlp_bwd(d, 10, 256, 256, 256, 256, 256, 256, None, 256, n, 0)
    assert e.value.status == 1
    with pytest.raises(g.MoeError) as e:
        g.mxfp8_quantize(256, 64, 40, 1, 0, 256, 256, None, None, 0)
    assert e.value.status == 2
    with pytest.raises(g.MoeError) as e:
        g.mxfp8_quantize(256, 48, 64, 0, 1, None, None, 256, 256, 0)
    assert e.value.status == 2
    with pytest.raises(g.MoeError) as e:
        g.moe_pack_fc1_weight(256, 256, 2, 64, 64, 1, 64, 0, 0)
    assert e.value.status == 1
    with pytest.raises(g.MoeError) as e:
        g.moe_pack_fc1_weight(256, 512, 2, 64, 96, 1, 64, 0, 0)
    assert e.value.status == 2
    assert "ilv" in lib.moe_last_error_string().decode()
    with pytest.raises(g.MoeError) as e:
        g.moe_selftest_wait_timeout(None, 10**8, 0)
    assert e.value.status == 1
    with pytest.raises(g.MoeError) as e:
        g.moe_selftest_wait_timeout(256, 10**3, 0)
    assert e.value.status == 1
    # the GEMM self-test: BF16 layers only, a w2 and a limit in [1 ms, 10 s], checked before
    # anything is enqueued
    mx = g.make_desc(E=4, k=2, H=128, F=128, T_max=16, precision="mxfp8", align=128)
    with pytest.raises(g.MoeError) as e:
        g.moe_selftest_gemm_timeout(mx, 256, 1 << 30, 256, 10**7, 0)
    assert e.value.status == 2
    bf = g.make_desc(E=4, k=2, H=128, F=128, T_max=16)
    with pytest.raises(g.MoeError) as e:
        g.moe_selftest_gemm_timeout(bf, 256, 1 << 30, None, 10**7, 0)
    assert e.value.status == 1
    with pytest.raises(g.MoeError) as e:
        g.moe_selftest_gemm_timeout(bf, 256, 1 << 30, 256, 10**3, 0)
    assert e.value.status == 1
    # route export: T within [0, T_max], 4-byte aligned destinations, a workspace
    with pytest.raises(g.MoeError) as e:
        g.moe_route_export(bf, 256, 1 << 30, 17, 256, 256, 256, 256, 0)
    assert e.value.status == 1
    with pytest.raises(g.MoeError) as e:
        g.moe_route_export(bf, 256, 1 << 30, 8, 258, None, None, None, 0)
    assert e.value.status == 1
    with pytest.raises(g.MoeError) as e:
        g.moe_route_export(bf, None, 1 << 30, 8, 256, None, None, None, 0)
    assert e.value.status == 1


def test_config_table_matches_workloads():
    c = synth.CONFIGS
    assert (c["mixtral_bf16"].T, c["mixtral_bf16"].E, c["mixtral_bf16"].k) == (8192, 8, 2)
    assert c["mixtral_bf16"].flops_fwd_bwd() == pytest.approx(1.732e13, rel=1e-3)
    assert c["tiny"].flops_fwd_bwd() == pytest.approx(6.04e8, rel=1e-3)
    assert c["dsv3_mxfp8"].R == 32768 and c["gptoss_bf16"].R == 65536
    for cfg in c.values():
        d = g.desc_from_config(cfg)
        assert d.H % 64 == 0 and d.F % 64 == 0
