"""Shared helpers for the tests: building the library, tolerances, comparisons."""

import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# Parity bar for attention outputs on unit-variance inputs (max-abs / mean-abs
# of fp16 O against the float64 oracle), and our bound on the natural-log lse.
O_MAX_ABS = 4e-3
O_MEAN_ABS = 5e-4
LSE_ABS = 1e-3


def ensure_library():
    """Build libqattn.so in-tree if it is missing or stale; return the module."""
    from quantized_kv_attention_gb300 import build
    build.build()
    import quantized_kv_attention_gb300 as qa
    qa.load_library()
    return qa


def header_symbols():
    """Function names declared in include/qattn.h."""
    with open(os.path.join(ROOT, "include", "qattn.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qattn_[a-z0-9_]+)\s*\(", text)))


def require_gpu():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return ensure_library()


def assert_close_attention(out_gpu, ref, what="O", max_abs=O_MAX_ABS, mean_abs=O_MEAN_ABS):
    o = out_gpu.detach().float().cpu().numpy().astype(np.float64)
    assert o.shape == ref.shape, (o.shape, ref.shape)
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    err = np.abs(o - ref)
    mx, mn = float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0
    assert mx <= max_abs and mn <= mean_abs, f"{what}: max-abs {mx:.3e} mean-abs {mn:.3e}"
    return mx, mn


def assert_close_lse(lse_gpu, ref, tol=LSE_ABS):
    l = lse_gpu.detach().cpu().numpy().astype(np.float64)
    fin = np.isfinite(ref)
    assert (np.isfinite(l) == fin).all(), "lse: finiteness differs"
    assert (l[~fin] == -np.inf).all()
    if fin.any():
        err = float(np.abs(l[fin] - ref[fin]).max())
        assert err <= tol, f"lse max-abs {err:.3e}"


# Out-of-bounds checks without compute-sanitizer: an output placed in the middle
# of a buffer whose margins (and body) hold a fixed bit pattern.
GUARD_MARGIN = 4096  # elements on each side (a multiple of 16 bytes for 2- and 4-byte types)
_GUARD_BITS = {2: 0x5A5A, 4: 0x5A5A5A5A}


def guarded(shape, dtype):
    """(buffer, view): a device tensor of `shape` and `dtype` inside a buffer whose
    margins hold the guard pattern; the tensor starts with the pattern too, so an
    element the call leaves unwritten shows."""
    import torch
    n = 1
    for d in shape:
        n *= int(d)
    size = torch.empty((), dtype=dtype).element_size()
    ity = {2: torch.int16, 4: torch.int32}[size]
    buf = torch.full((n + 2 * GUARD_MARGIN,), _GUARD_BITS[size], dtype=ity, device="cuda")
    return buf, buf[GUARD_MARGIN:GUARD_MARGIN + n].view(dtype).view(*shape)


def check_guards(buf, what, body_written=True):
    """The margins are untouched; with body_written, no element kept the pattern."""
    bits = _GUARD_BITS[buf.element_size()]
    n = buf.numel() - 2 * GUARD_MARGIN
    assert bool((buf[:GUARD_MARGIN] == bits).all()), f"{what}: a write before the output"
    assert bool((buf[GUARD_MARGIN + n:] == bits).all()), f"{what}: a write after the output"
    if body_written:
        assert not bool((buf[GUARD_MARGIN:GUARD_MARGIN + n] == bits).any()), f"{what}: elements left unwritten"


def mutant_fails_a_pin(monkeypatch, module, func_name, old, new, pins):
    """Plant a mistake in one oracle function (its source with `old` replaced by
    `new`, on the CPU) and report whether one of the pin tests `pins` fails."""
    import inspect
    import textwrap
    owner, attr = module, func_name
    if "." in func_name:  # a method: "Class.method"
        cls, attr = func_name.split(".")
        owner = getattr(module, cls)
    src = textwrap.dedent(inspect.getsource(getattr(owner, attr)))
    assert old in src, (func_name, old)
    ns = dict(vars(module))
    exec(compile(src.replace(old, new, 1), "<mutant>", "exec"), ns)
    monkeypatch.setattr(owner, attr, ns[attr])
    for pin in pins:
        try:
            pin()
        except (AssertionError, ValueError, IndexError, ZeroDivisionError, TypeError, OverflowError):
            return True
    return False
