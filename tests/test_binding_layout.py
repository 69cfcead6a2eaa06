"""The ctypes mirrors in the binding must lay out every struct of
``include/moe.h`` and ``include/moe_ep.h`` exactly as a C compiler does, and carry the header's enum
values.  A C probe is compiled against the header with the host compiler
(gcc or cc) and prints each struct's size and each field's offset, and each
enum constant.  Host code only: no GPU, no CUDA library needed.
"""

from __future__ import annotations

import ctypes
import os
import shutil
import subprocess

import pytest

from sparse_mixture_experts_softmax_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")

STRUCTS = {
    "moe_config": B.moe_config,
    "moe_weights": B.moe_weights,
    "moe_grads": B.moe_grads,
    "moe_params": B.moe_params,
    "moe_ep_config": B.moe_ep_config,
    "moe_ep_rows": B.moe_ep_rows,
}

ENUMS = {
    "MOE_OK": B.MOE_OK,
    "MOE_ERR_INVALID_ARG": B.MOE_ERR_INVALID_ARG,
    "MOE_ERR_UNSUPPORTED": B.MOE_ERR_UNSUPPORTED,
    "MOE_ERR_ALIGNMENT": B.MOE_ERR_ALIGNMENT,
    "MOE_ERR_WORKSPACE_TOO_SMALL": B.MOE_ERR_WORKSPACE_TOO_SMALL,
    "MOE_ERR_CUDA": B.MOE_ERR_CUDA,
    "MOE_ERR_TIMEOUT": B.MOE_ERR_TIMEOUT,
    "MOE_ACT_RELU": B.ACT["relu"],
    "MOE_ACT_GELU_TANH": B.ACT["gelu_tanh"],
    "MOE_ACT_SWIGLU": B.ACT["swiglu"],
    "MOE_SCORE_SOFTMAX": B.SCORE["softmax"],
    "MOE_SCORE_SIGMOID": B.SCORE["sigmoid"],
    "MOE_GROUP_TOP2_SUM": B.GROUP_SCORE["top2_sum"],
    "MOE_GROUP_MAX": B.GROUP_SCORE["max"],
    "MOE_F32": B.DTYPE["f32"],
    "MOE_BF16": B.DTYPE["bf16"],
    "MOE_GEMM_CUDA_CORES": B.GEMM_CUDA_CORES,
    "MOE_GEMM_TENSOR_BF16": B.GEMM_TENSOR_BF16,
    "MOE_GEMM_TENSOR_F32X3": B.GEMM_TENSOR_F32X3,
}


def _probe_source() -> str:
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "moe_ep.h"', "int main(void) {"]
    for name, cls in STRUCTS.items():
        lines.append(f'  printf("size {name} %zu\\n", sizeof({name}));')
        for field, ftype in cls._fields_:
            lines.append(f'  printf("offset {name}.{field} %zu\\n", offsetof({name}, {field}));')
            if issubclass(ftype, ctypes.Structure):
                # nested struct: its own fields are checked through STRUCTS
                continue
    for const in ENUMS:
        lines.append(f'  printf("enum {const} %d\\n", (int){const});')
    lines.append(f'  printf("define MOE_NOALLOC_MAX_ROUTED %d\\n", (int)MOE_NOALLOC_MAX_ROUTED);')
    lines += ["  return 0;", "}"]
    return "\n".join(lines) + "\n"


@pytest.fixture(scope="module")
def c_layout(tmp_path_factory):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no host C compiler")
    d = tmp_path_factory.mktemp("layout")
    src, exe = d / "probe.c", d / "probe"
    src.write_text(_probe_source())
    subprocess.run([cc, "-std=c11", "-Wall", "-Werror", "-I", HEADER_DIR, str(src), "-o", str(exe)],
                   check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    table = {}
    for line in out.splitlines():
        kind, key, value = line.split()
        table[(kind, key)] = int(value)
    return table


@pytest.mark.parametrize("name", sorted(STRUCTS))
def test_struct_layout_matches_header(c_layout, name):
    cls = STRUCTS[name]
    assert ctypes.sizeof(cls) == c_layout[("size", name)], f"sizeof({name})"
    for field, _ in cls._fields_:
        assert getattr(cls, field).offset == c_layout[("offset", f"{name}.{field}")], \
            f"offsetof({name}, {field})"


def test_field_lists_are_complete(c_layout):
    # every field of the C struct is mirrored: the last mirrored field ends
    # where the C struct ends (up to the struct's trailing alignment padding)
    for name, cls in STRUCTS.items():
        last, ltype = cls._fields_[-1]
        end = getattr(cls, last).offset + ctypes.sizeof(ltype)
        align = ctypes.alignment(cls)
        assert c_layout[("size", name)] - end < align, f"{name} has fields the binding lacks"


def test_enum_values_match_header(c_layout):
    for const, value in ENUMS.items():
        assert c_layout[("enum", const)] == value, const


def test_noalloc_limit_matches_header(c_layout):
    assert c_layout[("define", "MOE_NOALLOC_MAX_ROUTED")] == B.MOE_NOALLOC_MAX_ROUTED
