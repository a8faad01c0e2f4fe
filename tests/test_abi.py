"""The C-ABI library loads and exports every entry point include/eng.h declares (no GPU work)."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import synth
from harness import ensure_built

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "eng.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(eng_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_step_calls():
    names = declared_functions()
    for n in ["eng_create", "eng_capture", "eng_step", "eng_pool_alloc", "eng_pool_free", "eng_status",
              "eng_last_error", "eng_destroy"]:
        assert n in names


def test_library_exports_every_declared_symbol():
    eng = ensure_built()
    lib = eng.lib()
    for n in declared_functions():
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", eng.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (eng_[a-z_0-9]+)\b", out))
    assert set(declared_functions()) <= exported
    # the binding wraps every declared entry point under the same name
    assert {name for name, _, _ in eng.SIGNATURES} == set(declared_functions())


def test_struct_layouts_match_the_header(tmp_path):
    """Field offsets of the ctypes mirrors equal the C compiler's for include/eng.h."""
    eng = ensure_built()
    structs = {"eng_config_t": eng.eng_config_t, "eng_tensor_t": eng.eng_tensor_t, "eng_step_t": eng.eng_step_t,
               "eng_step_info_t": eng.eng_step_info_t}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "eng.h"', "int main(void) {"]
    for cname, cls in structs.items():
        lines.append(f'printf("{cname} size %zu\\n", sizeof({cname}));')
        for f, _ in cls._fields_:
            lines.append(f'printf("{cname} {f} %zu\\n", offsetof({cname}, {f}));')
    lines.append("return 0; }")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    for line in filter(None, out):
        cname, field, value = line.split()
        cls = structs[cname]
        want = ctypes.sizeof(cls) if field == "size" else getattr(cls, field).offset
        assert int(value) == want, line


def test_config_validation_rejects_bad_shapes_before_touching_a_device():
    eng = ensure_built()
    s = synth.shape("tiny")
    bad = [
        dict(head_dim=96),
        dict(kv_heads=3),
        dict(vocab=4100),
    ]
    for change in bad:
        cfg = eng.make_config(s, 16, 4, 64, 4)
        for k, v in change.items():
            setattr(cfg, k, v)
        with pytest.raises(eng.EngError) as ei:
            eng.eng_create(cfg, eng.TensorList([]), None)
        assert ei.value.code == eng.ENG_EINVAL
    cfg = eng.make_config(s, 16, 4, 64, 4)
    cfg.q_heads, cfg.kv_heads = 16, 1        # 16 query heads per KV head: beyond one MMA tile's hi/lo rows
    with pytest.raises(eng.EngError) as ei:
        eng.eng_create(cfg, eng.TensorList([]), None)
    assert ei.value.code == eng.ENG_EINVAL and "8 query heads" in str(ei.value)
    cfg = eng.make_config(s, 16, 4, 64, 4)
    cfg.block_size = 32
    with pytest.raises(eng.EngError) as ei:
        eng.eng_create(cfg, eng.TensorList([]), None)
    assert ei.value.code == eng.ENG_EINVAL and "block_size" in str(ei.value)
    cfg = eng.make_config(s, 16, 4, 64, 4)
    cfg.dtype = eng.ENG_DTYPE_F32             # matrices are 16-bit: bf16 or fp16
    with pytest.raises(eng.EngError) as ei:
        eng.eng_create(cfg, eng.TensorList([]), None)
    assert ei.value.code == eng.ENG_EINVAL and "dtype" in str(ei.value)


def test_binding_marks_the_16_bit_format():
    """make_config and TensorList carry the model's 16-bit format: bf16 (the default) or fp16."""
    eng = ensure_built()
    s = synth.shape("tiny")
    assert eng.make_config(s, 16, 4, 64, 4).dtype == eng.ENG_DTYPE_BF16
    assert eng.make_config(s, 16, 4, 64, 4, dtype="f16").dtype == eng.ENG_DTYPE_F16
    w = synth.make_weights(s, seed=0, dtype="f16")
    items = [(n, w[n]) for n in ("model.embed_tokens.weight", "model.norm.weight")]
    tl = eng.TensorList(items + [("x", np.zeros(4, np.float32))], "f16")
    assert [tl.array[i].dtype for i in range(tl.count)] == [eng.ENG_DTYPE_F16, eng.ENG_DTYPE_F16, eng.ENG_DTYPE_F32]
    assert eng.TensorList(items).array[0].dtype == eng.ENG_DTYPE_BF16
    with pytest.raises(ValueError):
        eng.make_config(s, 16, 4, 64, 4, dtype="f32")
    with pytest.raises(ValueError):
        eng.TensorList(items, "fp8")


def test_no_cpu_fallback_without_a_device():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    eng = ensure_built()
    s = synth.shape("tiny")
    with pytest.raises(eng.EngError) as ei:
        eng.eng_create(eng.make_config(s, 16, 4, 64, 4), eng.TensorList([]), None)
    assert ei.value.code == eng.ENG_ECUDA and "no CUDA device" in str(ei.value)


def test_null_arguments_are_rejected():
    eng = ensure_built()
    lib = eng.lib()
    assert lib.eng_step(None, None, None, None) == eng.ENG_EINVAL
    assert lib.eng_capture(None, None, 0) == eng.ENG_EINVAL
    assert lib.eng_status(None, 0) == eng.ENG_EINVAL
    lib.eng_destroy(None)
