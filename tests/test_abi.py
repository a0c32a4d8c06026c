"""The C ABI without a GPU: the library loads, exports what the header declares,
and rejects bad arguments before touching any device."""
import ctypes
import os
import re

import pytest

import dense_tiled_gemm_fp16_gb300 as g

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    src = open(os.path.join(ROOT, "include", "gemm_f16.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gemm_f16\w*)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    lib = g.lib()
    names = header_functions()
    assert set(names) == set(g.EXPORTED)
    for n in names:
        assert hasattr(lib, n), n
        assert ctypes.cast(getattr(lib, n), ctypes.c_void_p).value


def header_constants():
    """NAME -> value for every enum member and integer #define of the header."""
    src = open(os.path.join(ROOT, "include", "gemm_f16.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    out = {}
    for body in re.findall(r"enum\s*\{(.*?)\}", src, flags=re.S):
        for name, val in re.findall(r"(GEMM_F16_\w+)\s*=\s*(\d+)", body):
            out[name] = int(val)
    for name, expr in re.findall(r"#define\s+(GEMM_F16_\w+)\s+(.+)", src):
        expr = re.sub(r"\((?:int64_t|size_t)\)", "", expr).strip()
        if re.fullmatch(r"[\d\s()<]+", expr):
            out[name] = eval(expr)   # digits, parentheses and shifts only
    return out


def test_binding_constants_match_the_header():
    h = header_constants()
    prefix = "GEMM_F16_"
    for name, value in h.items():
        short = name[len(prefix):]
        if short.startswith(("OPT_", "ACT_", "ERR_")) or short == "OK":
            assert getattr(g, short) == value, name
    assert {v: k for k, v in h.items() if k.startswith(prefix + "ERR_") or k == prefix + "OK"} == g.STATUS
    assert g.MAX_DIM == h["GEMM_F16_MAX_DIM"]
    assert g.MAX_GROUPS == h["GEMM_F16_MAX_GROUPS"]
    assert g.NOALLOC_SCRATCH_BYTES == h["GEMM_F16_NOALLOC_SCRATCH_BYTES"]
    assert g.gemm_f16_abi_version() == h["GEMM_F16_ABI_VERSION"]
    assert len([k for k in h if k.startswith(prefix + "OPT_")]) == 19   # (12 is left unused)


def test_status_strings_and_version():
    assert g.gemm_f16_abi_version() == 3
    for code, name in g.STATUS.items():
        assert g.gemm_f16_status_string(code) == name
    assert g.gemm_f16_status_string(99) == "GEMM_F16_UNKNOWN_STATUS"


# Fake, non-null, 256-byte-aligned "pointers": validation rejects these calls
# before any CUDA call, so nothing is ever dereferenced.
A, B, C = 1 << 20, 1 << 24, 1 << 28


@pytest.mark.parametrize("args", [
    (0, 4, 1, B, 4, 1, C, 4, 4, 4, 4),        # null A
    (A, 4, 1, 0, 4, 1, C, 4, 4, 4, 4),        # null B
    (A, 4, 1, B, 4, 1, 0, 4, 4, 4, 4),        # null C
    (A, 4, 1, B, 4, 1, C, 4, 0, 4, 4),        # M = 0
    (A, 4, 1, B, 4, 1, C, 4, 4, 0, 4),        # N = 0
    (A, 4, 1, B, 4, 1, C, 4, 4, 4, 0),        # K = 0
    (A, 0, 1, B, 4, 1, C, 4, 4, 4, 4),        # zero stride (broadcast) is outside the contract
    (A, 4, -1, B, 4, 1, C, 4, 4, 4, 4),       # negative stride
    (A, 4, 1, B, 4, 1, C, 3, 4, 4, 4),        # ldc < N
    (A + 1, 4, 1, B, 4, 1, C, 4, 4, 4, 4),    # fp16 pointer not 2-byte aligned
    (A, 1 << 62, 1, B, 4, 1, C, 4, 4, 4, 4),  # extent overflows int64
    (A, 1 << 31, 1, B, 1, 1, C, 1, 1, 1, 1 << 31),            # K beyond the 32-bit copy coordinates
    (A, 1, 1, B, 1, 1, C, 1, g.MAX_DIM + 1, 1, 1),            # M one past the limit
    (A, 1, 1, B, 1, 1, C, g.MAX_DIM + 1, 1, g.MAX_DIM + 1, 1),  # N one past the limit
])
def test_invalid_arguments(args):
    with pytest.raises(g.GemmF16Error) as e:
        g.gemm_f16(*args)
    assert e.value.status == g.ERR_INVALID_VALUE


def test_largest_dimension_passes_validation():
    # M = N = 1, K at the limit: validation accepts it and, without a GB300,
    # the call stops at the device check
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    a, b, c = 1 << 20, 1 << 40, 1 << 44   # fake pointers whose 4 GB views do not overlap
    with pytest.raises(g.GemmF16Error) as e:
        g.gemm_f16(a, g.MAX_DIM, 1, b, 1, 1, c, 1, 1, 1, g.MAX_DIM)
    assert e.value.status == g.ERR_UNSUPPORTED_DEVICE


def test_grouped_total_rows_beyond_the_limit():
    half = g.MAX_DIM // 2 + 1
    with pytest.raises(g.GemmF16Error) as e:
        g.gemm_f16_grouped(A, 4, 1, B, 16, 4, 1, C, 4, [half, half], 4, 4)
    assert e.value.status == g.ERR_INVALID_VALUE


def test_alias_detected():
    # C's 4x4 view overlaps A's view
    with pytest.raises(g.GemmF16Error) as e:
        g.gemm_f16(A, 4, 1, B, 4, 1, A + 8, 4, 4, 4, 4)
    assert e.value.status == g.ERR_ALIAS
    # C inside B's span (a transposed B spanning K*sbn)
    with pytest.raises(g.GemmF16Error) as e:
        g.gemm_f16(A, 4, 1, B, 1, 1000, B + 2 * 500, 4, 4, 4, 4)
    assert e.value.status == g.ERR_ALIAS


def test_valid_arguments_reach_the_device_check():
    # On a host without a GB300 a well-formed call stops at the device check.
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(g.GemmF16Error) as e:
        g.gemm_f16(A, 4, 1, B, 4, 1, C, 4, 4, 4, 4)
    assert e.value.status == g.ERR_UNSUPPORTED_DEVICE


def test_options_validation():
    with pytest.raises(g.GemmF16Error):
        g.gemm_f16_set_option(99, 1)
    with pytest.raises(g.GemmF16Error):
        g.gemm_f16_set_option(g.OPT_TILE_N, 100)
    with pytest.raises(g.GemmF16Error):
        g.gemm_f16_set_option(g.OPT_SWAP, 3)
    with pytest.raises(g.GemmF16Error):
        g.gemm_f16_set_option(g.OPT_SPLITS, -1)
    g.gemm_f16_set_option(g.OPT_TILE_N, 128)
    g.gemm_f16_set_option(g.OPT_TILE_N, 0)


def test_package_has_no_oracle_dependency():
    # The product never imports the oracle.
    pkg = os.path.join(ROOT, "dense_tiled_gemm_fp16_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "gemm_oracle" not in text, f


# ------------------------------------------------ batched, grouped, fused
def test_batched_and_grouped_argument_errors():
    with pytest.raises(g.GemmF16Error) as e:   # batch 0
        g.gemm_f16_batched(A, 16, 4, 1, B, 16, 4, 1, C, 16, 4, 4, 4, 4, 0)
    assert e.value.status == g.ERR_INVALID_VALUE
    with pytest.raises(g.GemmF16Error) as e:   # the problems' outputs overlap (C stride below one view)
        g.gemm_f16_batched(A, 16, 4, 1, B, 16, 4, 1, C, 8, 4, 4, 4, 4, 2)
    assert e.value.status == g.ERR_INVALID_VALUE
    with pytest.raises(g.GemmF16Error) as e:   # a negative group
        g.gemm_f16_grouped(A, 4, 1, B, 16, 4, 1, C, 4, [3, -1], 4, 4)
    assert e.value.status == g.ERR_INVALID_VALUE
    with pytest.raises(g.GemmF16Error) as e:   # more groups than the limit
        g.gemm_f16_grouped(A, 4, 1, B, 16, 4, 1, C, 4, [1] * (g.MAX_GROUPS + 1), 4, 4)
    assert e.value.status == g.ERR_INVALID_VALUE
    # every group empty: nothing to do, no device touched
    g.gemm_f16_grouped(A, 4, 1, B, 16, 4, 1, C, 4, [0, 0, 0], 4, 4)


def test_fused_argument_errors_on_the_host():
    base = (A, 4, 1, B, 4, 1)
    with pytest.raises(g.GemmF16Error) as e:   # unknown activation
        g.gemm_f16_fused(*base, 0, 0, 0, 9, C, 4, 4, 4, 4)
    assert e.value.status == g.ERR_INVALID_VALUE
    with pytest.raises(g.GemmF16Error) as e:   # bias_up without an up projection
        g.gemm_f16_fused(*base, 0, 0, B + (1 << 12), 0, C, 4, 4, 4, 4)
    assert e.value.status == g.ERR_INVALID_VALUE
    with pytest.raises(g.GemmF16Error) as e:   # odd up-projection address
        g.gemm_f16_fused(*base, B + (1 << 12) + 1, 0, 0, 0, C, 4, 4, 4, 4)
    assert e.value.status == g.ERR_INVALID_VALUE
    with pytest.raises(g.GemmF16Error) as e:   # C overlaps the bias
        g.gemm_f16_fused(*base, 0, C + 2, 0, 1, C, 4, 4, 4, 4)
    assert e.value.status == g.ERR_ALIAS
    with pytest.raises(g.GemmF16Error) as e:   # C overlaps the up projection
        g.gemm_f16_fused(*base, C, 0, 0, 1, C, 4, 4, 4, 4)
    assert e.value.status == g.ERR_ALIAS
    with pytest.raises(g.GemmF16Error) as e:   # grouped: negative bias stride
        g.gemm_f16_grouped_fused(A, 4, 1, B, 16, 4, 1, 0, C + (1 << 12), 0, -1, 1, C, 4, [2, 2], 4, 4)
    assert e.value.status == g.ERR_INVALID_VALUE


@pytest.mark.parametrize("option,value", [(0, 0), (99, 0), (g.OPT_STREAMK, 3), (g.OPT_PAIR, 3), (g.OPT_SWAP, 3),
                                          (g.OPT_TILE_N, 96), (g.OPT_TILE_N, 320), (g.OPT_MAX_STAGES, 1),
                                          (12, 0), (12, 2), (g.OPT_L2_A, 4), (g.OPT_L2_C, 9), (g.OPT_TWO_K_LOADS, 2), (21, 0), (g.OPT_REPACK, 3), (g.OPT_PDL, 2),
                                          (g.OPT_DEBUG_BOUNDS, 3), (g.OPT_TEST_STALL, 2), (g.OPT_SPLITS, -1)])
def test_options_reject_values_out_of_range(option, value):
    with pytest.raises(g.GemmF16Error) as e:
        g.gemm_f16_set_option(option, value)
    assert e.value.status == g.ERR_INVALID_VALUE


def test_torch_wrappers_check_arguments_before_any_call():
    import torch
    a = torch.zeros((4, 8), dtype=torch.float16)
    b = torch.zeros((8, 6), dtype=torch.float16)
    with pytest.raises(ValueError):
        g.fused_mm(a, b, act="tanh")
    with pytest.raises(ValueError):                       # bias_up needs b_up
        g.fused_mm(a, b, bias_up=torch.zeros(6, dtype=torch.float16))
    with pytest.raises(ValueError):                       # b_up must have b's shape and strides
        g.fused_mm(a, b, b_up=torch.zeros((6, 8), dtype=torch.float16).t())
    with pytest.raises(ValueError):                       # a bias holds N values
        g.fused_mm(a, b, bias=torch.zeros(5, dtype=torch.float16))
    with pytest.raises(ValueError):                       # group rows must add up to a's rows
        g.grouped_mm(a, torch.zeros((2, 8, 6), dtype=torch.float16), [1, 2])
    with pytest.raises(ValueError):
        g.bmm(torch.zeros((2, 4, 8), dtype=torch.float16), torch.zeros((3, 8, 6), dtype=torch.float16))


def test_torch_wrappers_refuse_other_dtypes_shapes_and_devices():
    # The library reads raw fp16 device memory: a float32 tensor, an output of
    # the wrong shape or a host tensor is refused before any call.
    import torch
    h = torch.float16
    a, b = torch.zeros((4, 8), dtype=h), torch.zeros((8, 6), dtype=h)
    with pytest.raises(TypeError):
        g.matmul(a.float(), b)
    with pytest.raises(TypeError):                        # out of another dtype
        g.matmul(a, b, out=torch.zeros((4, 6)))
    with pytest.raises(ValueError):                       # out of another shape
        g.matmul(a, b, out=torch.zeros((4, 7), dtype=h))
    with pytest.raises(ValueError):                       # host tensors
        g.matmul(a, b)
    a3, b3 = torch.zeros((2, 4, 8), dtype=h), torch.zeros((2, 8, 6), dtype=h)
    with pytest.raises(ValueError):
        g.bmm(a3, b3, out=torch.zeros((2, 4, 5), dtype=h))
    with pytest.raises(TypeError):
        g.bmm(a3, b3.float())
    with pytest.raises(ValueError):
        g.fused_mm(a3, b3, out=torch.zeros((1, 4, 6), dtype=h))
    with pytest.raises(TypeError):
        g.fused_mm(a, b, out=torch.zeros((4, 6)))
    bg = torch.zeros((2, 8, 6), dtype=h)
    with pytest.raises(ValueError):
        g.grouped_mm(a, bg, [1, 3], out=torch.zeros((4, 7), dtype=h))
    with pytest.raises(TypeError):
        g.grouped_mm(a.float(), bg, [1, 3])
    with pytest.raises(ValueError):
        g.grouped_fused_mm(a, bg, [1, 3], act="tanh")
    with pytest.raises(ValueError):
        g.grouped_fused_mm(a, bg, [1, 3], out=torch.zeros((3, 6), dtype=h))
    with pytest.raises(ValueError):                       # host tensors
        g.grouped_fused_mm(a, bg, [1, 3])


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    # no fallback of any kind: without the built library every call raises
    monkeypatch.setattr(g, "_lib", None)
    monkeypatch.setattr(g, "LIB_PATH", str(tmp_path / "libgemm_f16.so"))
    with pytest.raises(g.GemmF16Error, match="not built"):
        g.lib()
    with pytest.raises(g.GemmF16Error):
        g.gemm_f16(A, 4, 1, B, 4, 1, C, 4, 4, 4, 4)


def test_plain_c_program_links_and_calls_the_library(tmp_path):
    # The boundary is a C ABI: a C11 program that includes the header, takes
    # the address of every declared function and calls the host-only ones
    # compiles, links against the library and runs without a GPU.
    import shutil
    import subprocess

    cc = shutil.which("gcc") or shutil.which("cc")
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    if cc is None or not os.path.exists(os.path.join(cuda_inc, "cuda_runtime_api.h")):
        pytest.skip("no C compiler or CUDA headers")
    g.lib()   # built
    names = header_functions()
    src = tmp_path / "use.c"
    src.write_text(
        "#include <stdio.h>\n#include \"gemm_f16.h\"\n"
        "int main(void) {\n"
        "    const void* fns[] = {" + ", ".join(f"(const void*){n}" for n in names) + "};\n"
        "    size_t i, live = 0;\n"
        "    for (i = 0; i < sizeof fns / sizeof fns[0]; ++i) live += fns[i] != 0;\n"
        "    printf(\"%zu %d %s\\n\", live, gemm_f16_abi_version(), gemm_f16_status_string(GEMM_F16_ERR_ALIAS));\n"
        "    return 0;\n}\n")
    exe = tmp_path / "use"
    libdir = os.path.dirname(g.LIB_PATH)
    subprocess.run([cc, "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-I", cuda_inc, str(src), "-L", libdir, "-lgemm_f16",
                    "-Wl,-rpath," + libdir, "-o", str(exe)], check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    assert out == [str(len(names)), "3", "GEMM_F16_ERR_ALIAS"]
