"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function the public headers declare, plans workspaces, and rejects bad
arguments before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_headers_declare_the_boundary():
    names = declared_functions()
    for required in ("fa_bwd", "fa_fwd", "fa_bwd_workspace_bytes", "fa_status_string"):
        assert required in names


def test_every_declared_symbol_is_exported(fa):
    L = fa.lib()
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing
    assert sorted(fa.EXPORTED) == declared_functions()


def test_status_strings(fa):
    for s in range(6):
        assert fa.status_string(s)
    assert fa.status_string(99) == "unknown status"


def test_workspace_planning(fa):
    # dense: rows = B * Hq * round_up(Sq, 128)
    n = fa.workspace_bytes(2, 8192, 8192, 32, 8, 128)
    lay = fa.workspace_layout(2, 8192, 8192, 32, 8, 128)
    assert lay["rows"] == 2 * 32 * 8192
    assert lay["dqacc"] * 4 + lay["rows"] * 128 * 4 <= n
    lay = fa.workspace_layout(1, 130, 130, 2, 2, 64)
    assert lay["rows"] == 1 * 2 * 256
    # varlen: rows_per_head = round_up(B * (Sq + 128), 128)
    lay = fa.workspace_layout(3, 300, 300, 4, 4, 64, varlen=True)
    assert lay["rows"] == 4 * ((3 * (300 + 128) + 127) // 128 * 128)
    assert fa.workspace_bytes(2, 100, 100, 4, 4, 128, deterministic=True) > \
        fa.workspace_bytes(2, 100, 100, 4, 4, 128)
    assert fa.workspace_bytes(1, 128, 128, 1, 1, 100) == 0         # unsupported head dim
    assert fa.workspace_bytes(1, 128, 128, 1, 1, 48) == 0
    # D = 96 runs at the 128 tile width: the same workspace as D = 128
    assert fa.workspace_bytes(1, 128, 128, 1, 1, 96) == fa.workspace_bytes(1, 128, 128, 1, 1, 128)
    assert fa.workspace_bytes(1, 128, 128, 3, 2, 64) == 0          # Hq % Hkv != 0
    assert fa.workspace_bytes(0, 128, 128, 1, 1, 64) == 0


def _call_with_ws(fa, **over):
    """fa_bwd_with_workspace with fake (never dereferenced) aligned pointers."""
    L = fa.lib()
    a = dict(q=0x1000, k=0x2000, v=0x3000, o=0x4000, dout=0x5000, lse=0x6000, dq=0x7000,
             dk=0x8000, dv=0x9000, B=1, Sq=128, Sk=128, Hq=2, Hkv=2, D=64, scale=0.125,
             causal=0, cu_q=None, cu_k=None, det=0, dtype=0, ws=0x100000, ws_bytes=1 << 40)
    a.update(over)
    vp = ctypes.c_void_p
    return L.fa_bwd_with_workspace(
        vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["o"]), vp(a["dout"]), vp(a["lse"]), vp(a["dq"]),
        vp(a["dk"]), vp(a["dv"]), a["B"], a["Sq"], a["Sk"], a["Hq"], a["Hkv"], a["D"],
        a["scale"], a["causal"], vp(a["cu_q"]) if a["cu_q"] else None,
        vp(a["cu_k"]) if a["cu_k"] else None, a["det"], a["dtype"], vp(a["ws"]), a["ws_bytes"],
        None)


@pytest.mark.parametrize("over,status", [
    (dict(q=0), 1), (dict(dv=0), 1), (dict(B=0), 1), (dict(Sq=-1), 1), (dict(Hq=3), 1),
    (dict(D=100), 2), (dict(D=264), 2), (dict(D=32), 2), (dict(dtype=7), 2),
    (dict(scale=0.0), 1), (dict(scale=float("nan")), 1), (dict(scale=float("inf")), 1),
    (dict(q=0x1008), 1), (dict(lse=0x6004), 1), (dict(ws=0x100010), 1), (dict(ws=0), 1),
    (dict(ws_bytes=16), 1), (dict(cu_q=0xA000), 1),
])
def test_invalid_arguments_rejected_before_launch(fa, over, status):
    assert _call_with_ws(fa, **over) == status


def test_fa_bwd_rejects_before_device(fa):
    L = fa.lib()
    vp = ctypes.c_void_p
    ptrs = [vp(0x1000 * (i + 1)) for i in range(9)]
    assert L.fa_bwd(*ptrs, 1, 128, 128, 3, 2, 64, 0.125, 0, None, None, 0, 0, None) == 1
    assert L.fa_bwd(*ptrs, 1, 128, 128, 2, 2, 84, 0.125, 0, None, None, 0, 0, None) == 2
    assert L.fa_fwd(*ptrs[:5], 1, 128, 128, 2, 2, 64, -1.0, 0, None, None, 0, None) == 1


def test_stage_entry_points_reject_null_tensors(fa):
    L = fa.lib()
    vp = ctypes.c_void_p
    ws = vp(0x100000)
    shape = (1, 128, 128, 2, 2, 64)
    # fa_bwd_main needs q, k, v, dout, dk, dv
    assert L.fa_bwd_main(vp(0x1000), vp(0x2000), vp(0x3000), None, vp(0x5000), vp(0x6000),
                         *shape, 0.125, 0, None, None, 0, 0, ws, 1 << 40, None) == 1
    assert L.fa_bwd_preprocess(vp(0x1000), None, vp(0x3000), *shape, None, None, 0, 0, ws,
                               1 << 40, None) == 1
    assert L.fa_bwd_postprocess(None, *shape, 0.125, None, None, 0, 0, ws, 1 << 40, None) == 1


def test_wait_timeout_setting(fa):
    old = fa.set_wait_timeout_ns(123456789)
    assert fa.set_wait_timeout_ns(0) == 123456789
    fa.set_wait_timeout_ns(old)


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    import attention_backward_preprocess_gb300 as mod
    monkeypatch.setattr(mod, "_lib", None)
    monkeypatch.setattr(mod, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no fallback"):
        mod.lib()


def test_fa_ext_layout_matches_the_header(fa, tmp_path):
    """The binding's FaExt has the size and field offsets of fa_ext in
    include/fa.h, as a C compiler lays it out."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    cuda_inc = None
    for d in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if d and os.path.exists(os.path.join(d, "include", "cuda_runtime_api.h")):
            cuda_inc = os.path.join(d, "include")
    if cc is None or cuda_inc is None:
        pytest.skip("no C compiler or CUDA headers")
    fields = [f[0] for f in fa.FaExt._fields_]
    src = tmp_path / "layout.c"
    src.write_text(
        "#include <stdio.h>\n#include <stddef.h>\n#include \"fa.h\"\n"
        "int main(void) {\n  printf(\"%zu\\n\", sizeof(fa_ext));\n" +
        "".join("  printf(\"%%zu\\n\", offsetof(fa_ext, %s));\n" % f for f in fields) +
        "  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", os.path.join(ROOT, "include"), "-I", cuda_inc, str(src), "-o",
                    str(exe)], check=True, capture_output=True)
    out = [int(x) for x in subprocess.run([str(exe)], check=True, capture_output=True,
                                          text=True).stdout.split()]
    assert out[0] == ctypes.sizeof(fa.FaExt)
    for f, off in zip(fields, out[1:]):
        assert getattr(fa.FaExt, f).offset == off, f


def test_dropout_mask_shape():
    import torch
    import attention_backward_preprocess_gb300 as m
    q = torch.empty(2, 300, 4, 64)
    k = torch.empty(2, 333, 2, 64)
    assert m.dropout_mask_shape(q, k) == (2, 4, 300, 11)
    qv = torch.empty(469, 4, 64)
    kv = torch.empty(469, 2, 64)
    cu = torch.tensor([0, 300, 429, 469], dtype=torch.int32)
    assert m.dropout_mask_shape(qv, kv, cu, 300) == (4, 469, 10)


# Extension arguments the library must refuse on the host, before it looks at
# the device (every case here fails validation, so nothing is launched).
EXT_BAD = [
    (dict(window_left=-2), 1),
    (dict(window_right=-5), 1),
    (dict(alibi_slopes=0x2000, alibi_batch_stride=3), 1),   # stride neither 0 nor Hq
    (dict(alibi_slopes=0x2002), 1),                         # slopes not 4-byte aligned
    (dict(seqused_q=0x2001), 1),
    (dict(dropout_p=1.0), 1),
    (dict(dropout_p=-0.25), 1),
    (dict(dropout_p=0.1, dropout_mask=0x3002), 1),          # mask not 4-byte aligned
    (dict(bias=0x4008), 1),                                 # bias not 16-byte aligned
]


def _fa_ext(fa, over):
    e = fa.FaExt(-1, -1, None, 0, None, None, None, 0, 0, 0, None, 0.0, 0, 0, None, 0, 0)
    for name, val in over.items():
        setattr(e, name, val)
    return e


@pytest.mark.parametrize("over,status", EXT_BAD, ids=lambda v: ",".join(v) if isinstance(v, dict) else "")
def test_extension_arguments_rejected_on_the_host(fa, over, status):
    L = fa.lib()
    vp = ctypes.c_void_p
    ptrs = [vp(0x1000 * (i + 1)) for i in range(9)]
    e = _fa_ext(fa, over)
    shape = (1, 128, 128, 2, 2, 64)
    assert L.fa_fwd_ext(*ptrs[:5], *shape, 0.125, 1, None, None, ctypes.byref(e), 0, None) == status
    assert L.fa_bwd_ext(*ptrs, *shape, 0.125, 1, None, None, ctypes.byref(e), 0, 0,
                        vp(0x100000), ctypes.c_size_t(1 << 40), None) == status


# packed totals given by the caller: varlen only, both positive, at most B * max
TOTALS_BAD = [
    (dict(total_q=100, total_k=100), False),          # a dense call
    (dict(total_q=100, total_k=0), True),             # one of the two missing
    (dict(total_q=-1, total_k=100), True),
    (dict(total_q=2 * 128 + 1, total_k=100), True),   # above B * Sq
    (dict(total_q=100, total_k=2 * 128 + 1), True),   # above B * Sk
]


@pytest.mark.parametrize("over,varlen", TOTALS_BAD, ids=[str(i) for i in range(len(TOTALS_BAD))])
def test_packed_totals_rejected_on_the_host(fa, over, varlen):
    L = fa.lib()
    vp = ctypes.c_void_p
    ptrs = [vp(0x1000 * (i + 1)) for i in range(9)]
    e = _fa_ext(fa, over)
    cu = vp(0x8000) if varlen else None
    shape = (2, 128, 128, 2, 2, 64)
    assert L.fa_fwd_ext(*ptrs[:5], *shape, 0.125, 1, cu, cu, ctypes.byref(e), 0, None) == 1
    assert L.fa_bwd_ext(*ptrs, *shape, 0.125, 1, cu, cu, ctypes.byref(e), 0, 0,
                        vp(0x100000), ctypes.c_size_t(1 << 40), None) == 1


@pytest.mark.parametrize("varlen", [False, True])
@pytest.mark.parametrize("det", [False, True])
def test_workspace_sync_layout(fa, varlen, det):
    """The error word opens the workspace; the semaphores (deterministic only)
    are one int32 per 64 workspace rows and lie inside the workspace, after
    the dQ accumulator."""
    shape = (3, 200, 300, 4, 2, 96)
    sync = fa.workspace_sync_layout(*shape, varlen=varlen, deterministic=det)
    lay = fa.workspace_layout(*shape, varlen=varlen, deterministic=det)
    total = fa.workspace_bytes(*shape, varlen=varlen, deterministic=det)
    assert sync["err"] == 0
    if det:
        assert sync["n_sem"] == lay["rows"] // 64
        assert sync["sem"] >= 4 * (lay["dqacc"] + lay["rows"] * 128)
        assert sync["sem"] % 4 == 0
        assert sync["sem"] + 4 * sync["n_sem"] <= total
    else:
        assert sync["sem"] == 0 and sync["n_sem"] == 0


# head dims: (D, Dv (0 = D), extension overrides, deterministic) -> status on the host
HEAD_DIMS = [
    ((264, 0), {}, 0, 2),          # D above 256
    ((56, 0), {}, 0, 2),           # D below 64
    ((100, 0), {}, 0, 2),          # not a multiple of 8
    ((64, 128), {}, 0, 2),         # Dv != D needs D > 64
    ((128, 4), {}, 0, 2),          # Dv below 8
    ((128, 260), {}, 0, 2),        # Dv above 256
    ((192, 0), {}, 1, 2),          # wide kernel: no deterministic order
    ((128, 96), dict(dropout_p=0.1), 0, 2),
    ((192, 0), dict(alibi_slopes=0x2000), 0, 2),
]


@pytest.mark.parametrize("dims,over,det,status", HEAD_DIMS,
                         ids=[str(i) for i in range(len(HEAD_DIMS))])
def test_head_dims_refused_on_the_host(fa, dims, over, det, status):
    L = fa.lib()
    vp = ctypes.c_void_p
    ptrs = [vp(0x1000 * (i + 1)) for i in range(9)]
    D, Dv = dims
    e = _fa_ext(fa, dict(over, head_dim_v=Dv))
    shape = (1, 128, 128, 2, 2, D)
    assert L.fa_bwd_ext(*ptrs, *shape, 0.125, 1, None, None, ctypes.byref(e), det, 0,
                        vp(0x100000), ctypes.c_size_t(1 << 40), None) == status


def test_wide_head_dim_workspace(fa):
    """The dQ accumulator runs at the tile width of D: 256 above 128."""
    for D, width in ((192, 256), (256, 256), (136, 256), (128, 128), (64, 64)):
        lay = fa.workspace_layout(1, 128, 128, 2, 2, D)
        n = fa.workspace_bytes(1, 128, 128, 2, 2, D)
        assert n >= 4 * (lay["dqacc"] + lay["rows"] * width)
        assert n < 4 * (lay["dqacc"] + lay["rows"] * width) + 4096


def test_d64_tile_width_follows_the_problem(fa):
    """D = 64 runs at the 128-wide tile for dense problems of 4096 keys or more
    (the accumulator is then 128 wide), at the 64-wide tile otherwise."""
    for Sk, varlen, width in ((4096, False, 128), (8192, False, 128), (4095, False, 64),
                              (8192, True, 64)):
        lay = fa.workspace_layout(2, Sk, Sk, 2, 2, 64, varlen=varlen)
        n = fa.workspace_bytes(2, Sk, Sk, 2, 2, 64, varlen=varlen)
        assert n >= 4 * (lay["dqacc"] + lay["rows"] * width)
        assert n < 4 * (lay["dqacc"] + lay["rows"] * width) + 4096


def test_stage_call_refusals(fa):
    """fa_bwd_stages_ext refuses an empty or unknown stage mask and a missing
    workspace before it touches the device."""
    L = fa.lib()
    vp = ctypes.c_void_p
    ptrs = [vp(0x1000 * (i + 1)) for i in range(9)]
    shape = (1, 128, 128, 2, 2, 64)
    for mask, ws in ((0, vp(0x100000)), (8, vp(0x100000)), (-1, vp(0x100000)), (7, None)):
        assert L.fa_bwd_stages_ext(mask, *ptrs, *shape, 0.125, 1, None, None, None, 0, 0, ws,
                                   ctypes.c_size_t(1 << 40), None) == fa.FA_ERR_INVALID_ARG


def test_bias_with_varlen_is_unsupported(fa):
    L = fa.lib()
    vp = ctypes.c_void_p
    ptrs = [vp(0x1000 * (i + 1)) for i in range(9)]
    e = _fa_ext(fa, dict(bias=0x4000, bias_row_stride=128))
    cu = vp(0x8000)
    assert L.fa_fwd_ext(*ptrs[:5], 2, 128, 128, 2, 2, 64, 0.125, 1, cu, cu, ctypes.byref(e), 0,
                        None) == 2


def test_forward_instance_choice(tmp_path):
    """The forward's instance choice (fa_fwd_common.h, host code): for every
    set of extensions a call needs, the instance picked has all of them and is
    the first such in the built list; the bias, dropout and D = 64 instances
    go to the two-warps-per-row kernel, the others to the one-warp kernel."""
    import shutil
    import subprocess
    cxx = shutil.which("g++") or shutil.which("c++")
    cuda_inc = None
    for d in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if d and os.path.exists(os.path.join(d, "include", "cuda.h")):
            cuda_inc = os.path.join(d, "include")
    if cxx is None or cuda_inc is None:
        pytest.skip("no C++ compiler or CUDA headers")
    csrc = os.path.join(ROOT, "attention_backward_preprocess_gb300", "csrc")
    src = tmp_path / "choice.cpp"
    src.write_text(
        # the header's inline helpers use CUDA's min / max; the host build
        # takes the standard ones
        '#include <cstdio>\n#include <algorithm>\nusing std::max;\nusing std::min;\n'
        '#include "fa_fwd_common.h"\n'
        "int main() {\n"
        "  for (int i = 0; i < fa::kNumFwdFlagSets; ++i) std::printf(\"set %d\\n\", fa::kFwdFlagSets[i]);\n"
        "  for (int need = 0; need < 16; need += 2)\n"
        "    std::printf(\"pick %d %d %d %d\\n\", need, fa::fwd_instance_flags(need),\n"
        "                fa::fwd_split(128, fa::fwd_instance_flags(need)),\n"
        "                fa::fwd_split(64, fa::fwd_instance_flags(need)));\n"
        "  return 0;\n}\n")
    exe = tmp_path / "choice"
    subprocess.run([cxx, "-std=c++17", "-I", csrc, "-I", os.path.join(ROOT, "include"), "-I",
                    cuda_inc, str(src), "-o", str(exe)], check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    sets = [int(ln.split()[1]) for ln in out if ln.startswith("set")]
    picks = [tuple(int(t) for t in ln.split()[1:]) for ln in out if ln.startswith("pick")]
    assert len(picks) == 8
    ALIBI, BIAS, DROP = 2, 4, 8
    for need, got, split128, split64 in picks:
        assert got & need == need
        assert got == next(s for s in sets if s & need == need)
        assert split128 == (1 if got & (BIAS | DROP) else 0)
        assert split64 == 1
