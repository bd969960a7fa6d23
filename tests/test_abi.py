"""The C ABI without a GPU: the library builds, loads, exports every function
include/kda.h declares, and rejects bad arguments on the host before any CUDA
call.  No kernel runs here."""
import ctypes

import pytest

import kimi_delta_attention_chunkwise_gb300 as kda
from kimi_delta_attention_chunkwise_gb300 import binding, build


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def test_header_declares_the_boundary():
    names = binding.header_functions()
    for required in ("kda_chunk_fwd", "kda_recurrent_step", "kda_status_string"):
        assert required in names


def test_library_exports_every_header_symbol(lib):
    for name in binding.header_functions():
        assert hasattr(lib, name), f"libkda.so does not export {name}"


def test_library_is_the_in_tree_build(lib):
    assert binding.lib_path().startswith(build.PKG)


def test_status_strings(lib):
    for code in range(5):
        s = kda.kda_status_string(code)
        assert s.startswith("KDA_")
    assert "UNKNOWN" in kda.kda_status_string(99)


def _shape(**kw):
    base = dict(N=1, T=64, H=2, dk=128, dv=128, dtype_code=kda.KDA_DTYPE_BF16)
    base.update(kw)
    return kda.make_shape(base["N"], base["T"], base["H"], base["dk"], base["dv"],
                          base["dtype_code"], base.get("chunk_size", 0),
                          base.get("engine", kda.KDA_ENGINE_AUTO))


FAKE = 0x10000  # 16-byte-aligned fake address: never dereferenced by these calls


def _chunk(lib, shape, ptrs=None, scale=1.0, cu=None):
    p = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, b=FAKE, out=FAKE)
    p.update(ptrs or {})
    return lib.kda_chunk_fwd(p["q"], p["k"], p["v"], p["g"], p["b"], ctypes.c_float(scale),
                             None, cu, p["out"], None,
                             ctypes.byref(shape) if shape is not None else None, None)


def test_chunk_rejects_bad_arguments(lib):
    assert _chunk(lib, None) == kda.KDA_ERR_INVALID_ARG
    assert _chunk(lib, _shape(N=0)) == kda.KDA_ERR_INVALID_ARG
    assert _chunk(lib, _shape(T=-1)) == kda.KDA_ERR_INVALID_ARG
    assert _chunk(lib, _shape(H=0)) == kda.KDA_ERR_INVALID_ARG
    assert _chunk(lib, _shape(dtype_code=7)) == kda.KDA_ERR_INVALID_ARG
    assert _chunk(lib, _shape(chunk_size=48)) == kda.KDA_ERR_INVALID_ARG
    assert _chunk(lib, _shape(engine=9)) == kda.KDA_ERR_INVALID_ARG
    assert _chunk(lib, _shape(N=3)) == kda.KDA_ERR_INVALID_ARG       # N > 1 needs cu_seqlens
    assert _chunk(lib, _shape(), scale=float("nan")) == kda.KDA_ERR_INVALID_ARG
    assert _chunk(lib, _shape(), ptrs={"v": FAKE + 2}) == kda.KDA_ERR_INVALID_ARG  # misaligned
    assert _chunk(lib, _shape(), ptrs={"b": FAKE + 2}) == kda.KDA_ERR_INVALID_ARG
    assert _chunk(lib, _shape(), ptrs={"out": None}) == kda.KDA_ERR_INVALID_ARG
    assert _chunk(lib, _shape(), ptrs={"g": None}) == kda.KDA_ERR_INVALID_ARG


def test_chunk_support_matrix(lib):
    assert _chunk(lib, _shape(dk=96, dv=96)) == kda.KDA_ERR_UNSUPPORTED
    assert _chunk(lib, _shape(dk=128, dv=64)) == kda.KDA_ERR_UNSUPPORTED
    # the tensor-core engine is bf16, d = 128, C = 64 only
    assert _chunk(lib, _shape(dtype_code=kda.KDA_DTYPE_F32,
                              engine=kda.KDA_ENGINE_TENSOR)) == kda.KDA_ERR_UNSUPPORTED
    assert _chunk(lib, _shape(dk=64, dv=64, engine=kda.KDA_ENGINE_TENSOR)) == kda.KDA_ERR_UNSUPPORTED
    assert _chunk(lib, _shape(chunk_size=32, engine=kda.KDA_ENGINE_TENSOR)) == kda.KDA_ERR_UNSUPPORTED


def test_workspace_query(lib):
    n = ctypes.c_size_t(123)
    assert lib.kda_chunk_fwd_workspace_size(None, ctypes.byref(n)) == kda.KDA_ERR_INVALID_ARG
    s = _shape(engine=kda.KDA_ENGINE_SIMT)
    assert lib.kda_chunk_fwd_workspace_size(ctypes.byref(s), ctypes.byref(n)) == kda.KDA_SUCCESS
    assert n.value == 0
    s = _shape(T=1 << 20, H=32)
    assert lib.kda_chunk_fwd_workspace_size(ctypes.byref(s), ctypes.byref(n)) == kda.KDA_SUCCESS
    assert n.value % 256 == 0


def test_workspace_variant_rejects_missing_scratch(lib):
    s = _shape(T=4096, H=16)
    need = ctypes.c_size_t(0)
    assert lib.kda_chunk_fwd_workspace_size(ctypes.byref(s), ctypes.byref(need)) == 0
    if need.value == 0:
        pytest.skip("engine needs no scratch")
    rc = lib.kda_chunk_fwd_ws(FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.c_float(1.0), None, None,
                              FAKE, None, ctypes.byref(s), None, 0, None)
    assert rc == kda.KDA_ERR_INVALID_ARG
    rc = lib.kda_chunk_fwd_ws(FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.c_float(1.0), None, None,
                              FAKE, None, ctypes.byref(s), FAKE + 16, need.value, None)
    assert rc == kda.KDA_ERR_INVALID_ARG  # not 256-byte aligned


def test_step_rejects_bad_arguments(lib):
    def step(shape, **kw):
        p = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, b=FAKE, s=FAKE, out=FAKE)
        p.update(kw)
        return lib.kda_recurrent_step(p["q"], p["k"], p["v"], p["g"], p["b"],
                                      ctypes.c_float(1.0), p["s"], p["out"],
                                      ctypes.byref(shape), None)
    assert step(_shape(N=4, T=5)) == kda.KDA_ERR_INVALID_ARG     # one token per sequence
    assert step(_shape(N=4, T=4), s=None) == kda.KDA_ERR_INVALID_ARG
    assert step(_shape(N=4, T=4), q=FAKE + 8) == kda.KDA_ERR_INVALID_ARG
    assert step(_shape(N=4, T=4), b=FAKE + 2) == kda.KDA_ERR_INVALID_ARG
    assert step(_shape(N=4, T=4, dk=48, dv=48)) == kda.KDA_ERR_UNSUPPORTED


def _recur(lib, shape, ptrs=None, cu=None, idx=None, num_slots=4, scale=1.0):
    p = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, b=FAKE, pool=FAKE, out=FAKE)
    p.update(ptrs or {})
    return lib.kda_recurrent_fwd(p["q"], p["k"], p["v"], p["g"], p["b"], ctypes.c_float(scale),
                                 cu, p["pool"], idx, num_slots, p["out"],
                                 ctypes.byref(shape) if shape is not None else None, None)


def test_recurrent_fwd_rejects_bad_arguments(lib):
    assert _recur(lib, None) == kda.KDA_ERR_INVALID_ARG
    assert _recur(lib, _shape(N=0)) == kda.KDA_ERR_INVALID_ARG
    assert _recur(lib, _shape(N=3)) == kda.KDA_ERR_INVALID_ARG            # N > 1 needs cu_seqlens
    assert _recur(lib, _shape(), num_slots=0) == kda.KDA_ERR_INVALID_ARG  # slot s for sequence s
    assert _recur(lib, _shape(), num_slots=-1, idx=FAKE) == kda.KDA_ERR_INVALID_ARG
    assert _recur(lib, _shape(), scale=float("inf")) == kda.KDA_ERR_INVALID_ARG
    assert _recur(lib, _shape(), ptrs={"pool": FAKE + 4}) == kda.KDA_ERR_INVALID_ARG
    assert _recur(lib, _shape(), ptrs={"pool": None}) == kda.KDA_ERR_INVALID_ARG
    assert _recur(lib, _shape(), idx=FAKE + 2) == kda.KDA_ERR_INVALID_ARG   # misaligned indices
    assert _recur(lib, _shape(dk=96, dv=96)) == kda.KDA_ERR_UNSUPPORTED


def test_value_head_groups_are_checked(lib):
    def shp(H, HV):
        return kda.make_shape(1, 64, H, 128, 128, kda.KDA_DTYPE_BF16, 0, kda.KDA_ENGINE_AUTO, 0, HV)
    assert _chunk(lib, shp(2, 3)) == kda.KDA_ERR_INVALID_ARG     # HV not a multiple of H
    assert _chunk(lib, shp(2, -2)) == kda.KDA_ERR_INVALID_ARG
    assert _recur(lib, shp(4, 6)) == kda.KDA_ERR_INVALID_ARG
    size = ctypes.c_size_t(0)
    assert lib.kda_chunk_fwd_workspace_size(ctypes.byref(shp(2, 8)), ctypes.byref(size)) == 0
    grouped = size.value
    assert lib.kda_chunk_fwd_workspace_size(ctypes.byref(shp(2, 0)), ctypes.byref(size)) == 0
    assert grouped == 4 * size.value or grouped > size.value   # scratch follows the value heads


def test_short_conv_rejects_bad_arguments(lib):
    def cs(N=1, T=16, C=64, W=4, dtype=kda.KDA_DTYPE_BF16, act=0):
        return kda.kdaConvShape_t(N, T, C, W, dtype, act)
    def fwd(shape, x=FAKE, w=FAKE, y=FAKE + 4096, cu=None):
        return lib.kda_short_conv_fwd(x, w, None, cu, None, None, y,
                                      ctypes.byref(shape) if shape is not None else None, None)
    assert fwd(None) == kda.KDA_ERR_INVALID_ARG
    assert fwd(cs(N=0)) == kda.KDA_ERR_INVALID_ARG
    assert fwd(cs(N=2)) == kda.KDA_ERR_INVALID_ARG          # N > 1 needs cu_seqlens
    assert fwd(cs(act=2)) == kda.KDA_ERR_INVALID_ARG
    assert fwd(cs(), y=FAKE) == kda.KDA_ERR_INVALID_ARG     # y must not be x
    assert fwd(cs(), x=FAKE + 8) == kda.KDA_ERR_INVALID_ARG  # 16-byte alignment
    assert fwd(cs(), w=None) == kda.KDA_ERR_INVALID_ARG
    assert fwd(cs(W=9)) == kda.KDA_ERR_UNSUPPORTED
    assert fwd(cs(C=60)) == kda.KDA_ERR_UNSUPPORTED
    assert lib.kda_short_conv_step(FAKE, FAKE, None, None, FAKE, ctypes.byref(cs()),
                                   None) == kda.KDA_ERR_INVALID_ARG   # no cache


def test_prologue_flags_are_checked(lib):
    def shp(pro, gb=None, ga=None):
        return kda.make_shape(1, 64, 2, 128, 128, kda.KDA_DTYPE_BF16, prologue=pro,
                              gate_bias=gb, gate_A_log=ga)
    assert _chunk(lib, shp(8)) == kda.KDA_ERR_INVALID_ARG                  # unknown bit
    assert _chunk(lib, shp(kda.KDA_PROLOGUE_GATE)) == kda.KDA_ERR_INVALID_ARG   # gate needs params
    assert _chunk(lib, shp(kda.KDA_PROLOGUE_GATE, FAKE, FAKE + 2)) == kda.KDA_ERR_INVALID_ARG
    assert _recur(lib, shp(kda.KDA_PROLOGUE_GATE, FAKE, None)) == kda.KDA_ERR_INVALID_ARG


def test_recurrent_bwd_support(lib):
    def bwd(shape):
        p = [FAKE] * 5
        return lib.kda_recurrent_bwd(p[0], p[1], p[2], p[3], p[4], ctypes.c_float(1.0), None, None,
                                     None, None, FAKE, FAKE, FAKE, FAKE, FAKE, None,
                                     ctypes.byref(shape), None)
    grouped = kda.make_shape(1, 64, 2, 128, 128, kda.KDA_DTYPE_BF16, num_v_heads=4)
    assert bwd(grouped) == kda.KDA_ERR_UNSUPPORTED
    pro = kda.make_shape(1, 64, 2, 128, 128, kda.KDA_DTYPE_BF16, prologue=kda.KDA_PROLOGUE_BETA_LOGITS)
    assert bwd(pro) == kda.KDA_ERR_UNSUPPORTED
    assert bwd(kda.make_shape(2, 64, 2, 128, 128, kda.KDA_DTYPE_BF16)) == kda.KDA_ERR_INVALID_ARG


def test_chunk_backward_workspace_variant_checks_its_scratch(lib):
    """kda_chunk_bwd_ws: the size query answers for the shapes the chunk form
    accepts, and missing, short or misaligned scratch is rejected before
    anything runs."""
    ok = kda.make_shape(1, 4096, 16, 128, 128, kda.KDA_DTYPE_BF16)
    n = ctypes.c_size_t(0)
    assert lib.kda_chunk_bwd_workspace_size(ctypes.byref(ok), ctypes.byref(n)) == kda.KDA_SUCCESS
    assert n.value > 0
    f32 = kda.make_shape(1, 4096, 16, 128, 128, kda.KDA_DTYPE_F32)
    assert lib.kda_chunk_bwd_workspace_size(ctypes.byref(f32), ctypes.byref(n)) == \
        kda.KDA_ERR_UNSUPPORTED
    need = ctypes.c_size_t(0)
    lib.kda_chunk_bwd_workspace_size(ctypes.byref(ok), ctypes.byref(need))

    def bwd_ws(ws, nbytes):
        return lib.kda_chunk_bwd_ws(FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.c_float(1.0), None, None,
                                    None, None, FAKE, FAKE, FAKE, FAKE, FAKE, None,
                                    ctypes.byref(ok), ws, ctypes.c_size_t(nbytes), None)
    assert bwd_ws(None, need.value) == kda.KDA_ERR_INVALID_ARG
    assert bwd_ws(FAKE, need.value - 1) == kda.KDA_ERR_INVALID_ARG
    assert bwd_ws(FAKE + 16, need.value) == kda.KDA_ERR_INVALID_ARG   # not 256-byte aligned


def test_chunk_bwd_support(lib):
    """The chunkwise backward takes bf16, d = 128 only, and checks the
    alignment its tensor maps need before anything runs."""
    def bwd(shape, q=FAKE):
        return lib.kda_chunk_bwd(q, FAKE, FAKE, FAKE, FAKE, ctypes.c_float(1.0), None, None,
                                 None, None, FAKE, FAKE, FAKE, FAKE, FAKE, None,
                                 ctypes.byref(shape), None)
    assert bwd(kda.make_shape(1, 64, 2, 128, 128, kda.KDA_DTYPE_F32)) == kda.KDA_ERR_UNSUPPORTED
    assert bwd(kda.make_shape(1, 64, 2, 64, 64, kda.KDA_DTYPE_BF16)) == kda.KDA_ERR_UNSUPPORTED
    grouped = kda.make_shape(1, 64, 2, 128, 128, kda.KDA_DTYPE_BF16, num_v_heads=4)
    assert bwd(grouped) == kda.KDA_ERR_UNSUPPORTED
    pro = kda.make_shape(1, 64, 2, 128, 128, kda.KDA_DTYPE_BF16, prologue=kda.KDA_PROLOGUE_L2NORM_QK)
    assert bwd(pro) == kda.KDA_ERR_UNSUPPORTED
    ok = kda.make_shape(1, 64, 2, 128, 128, kda.KDA_DTYPE_BF16)
    assert bwd(ok, q=FAKE + 4) == kda.KDA_ERR_INVALID_ARG      # q not 16-byte aligned
    assert bwd(kda.make_shape(2, 64, 2, 128, 128, kda.KDA_DTYPE_BF16)) == kda.KDA_ERR_INVALID_ARG


def test_chunk_backward_workspace_variant_checks_its_scratch(lib):
    """kda_chunk_bwd_ws: the size query answers for the shapes the chunk form
    accepts, and missing, short or misaligned scratch is rejected before
    anything runs."""
    ok = kda.make_shape(1, 4096, 16, 128, 128, kda.KDA_DTYPE_BF16)
    n = ctypes.c_size_t(0)
    assert lib.kda_chunk_bwd_workspace_size(ctypes.byref(ok), ctypes.byref(n)) == kda.KDA_SUCCESS
    assert n.value > 0
    f32 = kda.make_shape(1, 4096, 16, 128, 128, kda.KDA_DTYPE_F32)
    assert lib.kda_chunk_bwd_workspace_size(ctypes.byref(f32), ctypes.byref(n)) == \
        kda.KDA_ERR_UNSUPPORTED
    need = ctypes.c_size_t(0)
    lib.kda_chunk_bwd_workspace_size(ctypes.byref(ok), ctypes.byref(need))

    def bwd_ws(ws, nbytes):
        return lib.kda_chunk_bwd_ws(FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.c_float(1.0), None, None,
                                    None, None, FAKE, FAKE, FAKE, FAKE, FAKE, None,
                                    ctypes.byref(ok), ws, ctypes.c_size_t(nbytes), None)
    assert bwd_ws(None, need.value) == kda.KDA_ERR_INVALID_ARG
    assert bwd_ws(FAKE, need.value - 1) == kda.KDA_ERR_INVALID_ARG
    assert bwd_ws(FAKE + 16, need.value) == kda.KDA_ERR_INVALID_ARG   # not 256-byte aligned


def _align256(n):
    return (n + 255) // 256 * 256


def test_host_scratch_size_is_copies_plus_workspace(lib):
    """kda_chunk_fwd_host's scratch: a device copy of every input and output
    (each 256-byte aligned), then the engine's workspace."""
    T, H, d, N = 4096, 16, 128, 1
    s = _shape(T=T, H=H)
    ws, host = ctypes.c_size_t(0), ctypes.c_size_t(0)
    assert lib.kda_chunk_fwd_workspace_size(ctypes.byref(s), ctypes.byref(ws)) == kda.KDA_SUCCESS
    assert lib.kda_chunk_fwd_host_scratch_size(ctypes.byref(s), ctypes.byref(host)) == kda.KDA_SUCCESS
    tok = T * H * d
    regions = [2 * tok, 2 * tok, 2 * tok,        # q, k, v (bf16)
               4 * tok, 4 * T * H,               # log_alpha, beta
               4 * (N + 1),                      # cu_seqlens
               4 * N * H * d * d,                # initial state
               2 * tok,                          # out (bf16)
               4 * N * H * d * d]                # final state
    assert host.value == sum(_align256(r) for r in regions) + _align256(ws.value)
    assert lib.kda_chunk_fwd_host_scratch_size(None, ctypes.byref(host)) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_chunk_fwd_host_scratch_size(ctypes.byref(s), None) == kda.KDA_ERR_INVALID_ARG


def test_host_entry_rejects_bad_arguments(lib):
    """Every check runs on the host before any copy is enqueued."""
    s = _shape(T=4096, H=16)
    need = ctypes.c_size_t(0)
    assert lib.kda_chunk_fwd_host_scratch_size(ctypes.byref(s), ctypes.byref(need)) == 0

    def call(shape, scratch=FAKE, nbytes=None, **ptrs):
        p = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, b=FAKE, out=FAKE, cu=None)
        p.update(ptrs)
        return lib.kda_chunk_fwd_host(
            p["q"], p["k"], p["v"], p["g"], p["b"], ctypes.c_float(1.0), None, p["cu"],
            p["out"], None, ctypes.byref(shape) if shape is not None else None, scratch,
            need.value if nbytes is None else nbytes, None)

    assert call(None) == kda.KDA_ERR_INVALID_ARG
    assert call(s, scratch=None) == kda.KDA_ERR_INVALID_ARG
    assert call(s, nbytes=need.value - 256) == kda.KDA_ERR_INVALID_ARG
    assert call(s, scratch=FAKE + 16) == kda.KDA_ERR_INVALID_ARG    # not 256-byte aligned
    assert call(s, q=None) == kda.KDA_ERR_INVALID_ARG
    assert call(s, out=None) == kda.KDA_ERR_INVALID_ARG
    assert call(_shape(N=3, T=4096, H=16)) == kda.KDA_ERR_INVALID_ARG   # N > 1 needs cu_seqlens
    assert call(_shape(dk=96, dv=96)) == kda.KDA_ERR_UNSUPPORTED


# ---------------------------------------------------------------------------
# the binding against the header: prototypes and struct layouts
# ---------------------------------------------------------------------------

def _header_prototypes():
    """{name: (return type, [parameter declarations])} for every function
    include/kda.h declares."""
    import os
    import re
    with open(os.path.join(build.INCLUDE, "kda.h")) as f:
        text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
    protos = {}
    for m in re.finditer(r"(kdaStatus_t|const\s+char\s*\*)\s*(kda_\w+)\s*\(([^)]*)\)\s*;", text):
        params = [p.strip() for p in m.group(3).split(",") if p.strip() not in ("", "void")]
        protos[m.group(2)] = (m.group(1), params)
    return protos


def _c_kind(decl: str) -> str:
    if "*" in decl or "[" in decl or "cudaStream_t" in decl:
        return "pointer"
    if decl.startswith("float"):
        return "float"
    if "size_t" in decl:
        return "size"
    if decl.split()[0] in ("int32_t", "int", "kdaStatus_t", "kdaDtype_t"):
        return "int32"
    if decl.split()[0] == "int64_t":
        return "int64"
    raise AssertionError(f"unclassified parameter {decl!r}")


def _ctypes_kind(t) -> str:
    if t in (ctypes.c_void_p, ctypes.c_char_p) or issubclass(t, ctypes._Pointer):
        return "pointer"
    if t is ctypes.c_float:
        return "float"
    if t is ctypes.c_size_t:
        return "size"
    if t in (ctypes.c_int32, ctypes.c_int):
        return "int32"
    if t is ctypes.c_int64:
        return "int64"
    raise AssertionError(f"unclassified ctypes type {t!r}")


def test_binding_prototypes_match_the_header(lib):
    """Every declared function has a ctypes prototype with the same number
    and kinds of parameters (pointer, float, int32, size_t) and the same
    return kind, so no call marshals an argument into the wrong slot."""
    protos = _header_prototypes()
    assert set(protos) == set(binding.header_functions())
    for name, (ret, params) in protos.items():
        fn = getattr(lib, name)
        assert fn.argtypes is not None, f"{name}: no ctypes prototype"
        want = [_c_kind(p) for p in params]
        got = [_ctypes_kind(t) for t in fn.argtypes]
        assert got == want, f"{name}: binding {got} vs header {want}"
        if ret == "kdaStatus_t":
            assert fn.restype is ctypes.c_int, name
        else:
            assert fn.restype is ctypes.c_char_p, name


def test_struct_layouts_match_the_header(tmp_path):
    """kdaShape_t and kdaConvShape_t as the C compiler lays them out (a probe
    built with gcc against include/kda.h) equal the ctypes structures: the
    same size and the same offset and size for every field."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    cuda_inc = "/usr/local/cuda/include"
    import os
    if not gcc or not os.path.exists(os.path.join(cuda_inc, "cuda_runtime_api.h")):
        pytest.skip("gcc or the CUDA headers are missing")
    structs = {"kdaShape_t": binding.kdaShape_t, "kdaConvShape_t": binding.kdaConvShape_t}
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "kda.h"', "int main(void) {"]
    for sname, cls in structs.items():
        lines.append(f'  printf("{sname} . %zu %zu\\n", (size_t)0, sizeof({sname}));')
        for fname, _ in cls._fields_:
            lines.append(f'  printf("{sname} {fname} %zu %zu\\n", offsetof({sname}, {fname}), '
                         f'sizeof((({sname} *)0)->{fname}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([gcc, "-std=c99", "-I", build.INCLUDE, "-I", cuda_inc, str(src), "-o",
                    str(exe)], check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    seen = {}
    for line in out.splitlines():
        sname, fname, off, size = line.split()
        seen[(sname, fname)] = (int(off), int(size))
    for sname, cls in structs.items():
        assert seen[(sname, ".")][1] == ctypes.sizeof(cls), sname
        for fname, ftype in cls._fields_:
            assert seen[(sname, fname)] == (getattr(cls, fname).offset, ctypes.sizeof(ftype)), \
                (sname, fname)
