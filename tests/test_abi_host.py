"""The C-ABI library builds for sm_103a, loads without a GPU, exports every symbol
the header declares, and rejects bad arguments on the host (no kernel runs)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lp_ragged.h")

LP_OK, LP_ERR_NULL, LP_ERR_LEVELS, LP_ERR_SHAPE = 0, 1, 2, 3
LP_ERR_OFFSETS, LP_ERR_TOKEN_RANGE, LP_ERR_WORKSPACE, LP_ERR_CUDA = 4, 5, 6, 7
LP_ERR_TEMPERATURE = 8
FAKE = 0x10000          # non-NULL, 256-byte aligned, never dereferenced: each call returns first


@pytest.fixture(scope="module")
def lib():
    from ragged_log_probs_gb300 import _build
    _build.build()
    import ragged_log_probs_gb300 as lp
    return lp.load()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(lp_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    assert set(declared_functions()) >= {"lp_ragged_workspace_size", "lp_ragged_plan", "lp_ragged_compute",
                                         "lp_ragged_compute_ex", "lp_ragged_step", "lp_ragged_read_status",
                                         "lp_ragged_strerror"}


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_strerror_covers_codes(lib):
    seen = set()
    for code in range(LP_ERR_TEMPERATURE + 1):
        s = lib.lp_ragged_strerror(code).decode()
        assert s and s != "unknown lp_status"
        seen.add(s)
    assert len(seen) == LP_ERR_TEMPERATURE + 1
    assert lib.lp_ragged_strerror(99).decode() == "unknown lp_status"


def _compute(lib, logits=FAKE, T=4, V=100, off=FAKE, B=2, tokens=FAKE, sampled=FAKE, out_off=FAKE, echo=FAKE,
             levels=3, out_lp=FAKE, out_tok=FAKE, ws=FAKE, ws_bytes=1 << 20):
    return lib.lp_ragged_compute(logits, T, V, off, B, tokens, sampled, out_off, echo, levels, out_lp, out_tok,
                                 ws, ws_bytes, None)


def test_compute_host_checks(lib):
    assert _compute(lib, logits=None) == LP_ERR_NULL
    assert _compute(lib, tokens=None) == LP_ERR_NULL
    assert _compute(lib, out_tok=None) == LP_ERR_NULL
    assert _compute(lib, ws=None) == LP_ERR_WORKSPACE
    assert _compute(lib, levels=7) == LP_ERR_LEVELS
    assert _compute(lib, V=0) == LP_ERR_SHAPE
    assert _compute(lib, B=0) == LP_ERR_SHAPE
    assert _compute(lib, T=0) == LP_ERR_SHAPE
    assert _compute(lib, V=0x7FFFFFFF) == LP_ERR_SHAPE
    assert _compute(lib, logits=FAKE + 2) == LP_ERR_SHAPE
    assert _compute(lib, ws=FAKE + 16) == LP_ERR_WORKSPACE


def _compute_ex(lib, logits=FAKE, T_logits=4, V=100, loff=FAKE, ioff=None, T=4, B=2, tokens=FAKE, sampled=FAKE,
                out_off=FAKE, echo=FAKE, tau=None, levels=3, out_lp=FAKE, out_tok=FAKE, ws=FAKE, ws_bytes=1 << 20):
    return lib.lp_ragged_compute_ex(logits, T_logits, V, loff, ioff, T, B, tokens, sampled, out_off, echo, tau,
                                    levels, out_lp, out_tok, ws, ws_bytes, None)


def test_compute_ex_host_checks(lib):
    assert _compute_ex(lib, logits=None) == LP_ERR_NULL
    assert _compute_ex(lib, loff=None) == LP_ERR_NULL
    assert _compute_ex(lib, sampled=None) == LP_ERR_NULL
    assert _compute_ex(lib, ws=None) == LP_ERR_WORKSPACE
    assert _compute_ex(lib, levels=7) == LP_ERR_LEVELS
    assert _compute_ex(lib, T=6) == LP_ERR_SHAPE              # no input offsets: T must equal T_logits
    assert _compute_ex(lib, ioff=FAKE, T_logits=0) == LP_ERR_SHAPE
    assert _compute_ex(lib, ioff=FAKE, T=0) == LP_ERR_SHAPE
    assert _compute_ex(lib, V=0) == LP_ERR_SHAPE
    assert _compute_ex(lib, logits=FAKE + 1) == LP_ERR_SHAPE
    assert _compute_ex(lib, ws=FAKE + 64) == LP_ERR_WORKSPACE


def _step(lib, logits=FAKE, T_logits=4, V=100, loff=FAKE, ioff=None, T=4, B=2, tokens=FAKE, sampled=FAKE, echo=FAKE,
          tau=None, levels=3, out_off=FAKE, host=None, out_lp=FAKE, out_tok=FAKE, rows=4, ws=FAKE, ws_bytes=1 << 20):
    return lib.lp_ragged_step(logits, T_logits, V, loff, ioff, T, B, tokens, sampled, echo, tau, levels, out_off,
                              host, out_lp, out_tok, rows, ws, ws_bytes, None)


def test_step_host_checks(lib):
    # every check of the plan and the reduction comes before either launch
    assert _step(lib, rows=0) == LP_ERR_SHAPE
    assert _step(lib, logits=None) == LP_ERR_NULL
    assert _step(lib, loff=None) == LP_ERR_NULL
    assert _step(lib, out_off=None) == LP_ERR_NULL
    assert _step(lib, echo=None) == LP_ERR_NULL
    assert _step(lib, out_tok=None) == LP_ERR_NULL
    assert _step(lib, ws=None) == LP_ERR_WORKSPACE
    assert _step(lib, levels=7) == LP_ERR_LEVELS
    assert _step(lib, T=6) == LP_ERR_SHAPE                    # no input offsets: T must equal T_logits
    assert _step(lib, B=0) == LP_ERR_SHAPE
    assert _step(lib, V=0) == LP_ERR_SHAPE
    assert _step(lib, logits=FAKE + 1) == LP_ERR_SHAPE
    assert _step(lib, ws=FAKE + 64) == LP_ERR_WORKSPACE


def test_shard_entry_points_host_checks(lib):
    assert lib.lp_ragged_tuple_bytes(3) == 80 and lib.lp_ragged_tuple_bytes(6) == 528
    assert lib.lp_ragged_tuple_bytes(0) == 16 and lib.lp_ragged_tuple_bytes(7) == 0
    part = lambda **kw: lib.lp_ragged_shard_partials(
        kw.get("logits", FAKE), 4, kw.get("V", 100), kw.get("base", 0), FAKE, None, 4, 2, FAKE, FAKE, FAKE, FAKE,
        None, kw.get("levels", 3), kw.get("tuples", FAKE), kw.get("cap", 8), FAKE, 1 << 20, None)
    assert part(tuples=None) == LP_ERR_NULL
    assert part(tuples=FAKE + 8) == LP_ERR_SHAPE
    assert part(cap=0) == LP_ERR_SHAPE
    assert part(base=0x7FFFFFF0, V=100) == LP_ERR_SHAPE
    assert part(logits=None) == LP_ERR_NULL
    assert part(levels=7) == LP_ERR_LEVELS
    merge = lambda **kw: lib.lp_ragged_shard_merge(
        kw.get("tuples", FAKE), kw.get("P", 2), kw.get("cap", 8), kw.get("V", 100), FAKE, 2, None,
        kw.get("levels", 3), FAKE, FAKE, kw.get("ws", FAKE), 1 << 20, None)
    assert merge(tuples=None) == LP_ERR_NULL
    assert merge(ws=None) == LP_ERR_WORKSPACE
    assert merge(levels=7) == LP_ERR_LEVELS
    assert merge(P=0) == LP_ERR_SHAPE
    assert merge(V=0) == LP_ERR_SHAPE
    assert merge(cap=0) == LP_ERR_SHAPE
    assert merge(tuples=FAKE + 4) == LP_ERR_SHAPE


def test_plan_host_checks(lib):
    plan = lib.lp_ragged_plan
    assert plan(None, FAKE, 2, 4, FAKE, None, FAKE, 1 << 20, None) == LP_ERR_NULL
    assert plan(FAKE, None, 2, 4, FAKE, None, FAKE, 1 << 20, None) == LP_ERR_NULL
    assert plan(FAKE, FAKE, 2, 4, None, None, FAKE, 1 << 20, None) == LP_ERR_NULL
    assert plan(FAKE, FAKE, 2, 4, FAKE, None, None, 1 << 20, None) == LP_ERR_WORKSPACE
    assert plan(FAKE, FAKE, 0, 4, FAKE, None, FAKE, 1 << 20, None) == LP_ERR_SHAPE
    assert plan(FAKE, FAKE, 2, 0, FAKE, None, FAKE, 1 << 20, None) == LP_ERR_SHAPE


def test_read_status_and_workspace_size_host_checks(lib):
    assert lib.lp_ragged_read_status(None, FAKE, None) == LP_ERR_NULL
    assert lib.lp_ragged_read_status(FAKE, None, None) == LP_ERR_NULL
    assert lib.lp_ragged_workspace_size(2, 4, 100, 7) == 0


def test_package_fails_loudly_without_library(monkeypatch, tmp_path):
    import ragged_log_probs_gb300 as lp
    monkeypatch.setattr(lp, "_LIB", None)
    monkeypatch.setattr(lp._build, "lib_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        lp.load()


def test_binding_refuses_host_buffers_before_any_launch(lib):
    # The kernels write the workspace and read every array: host tensors are refused in the
    # binding, before a pointer reaches the library.
    import torch
    import ragged_log_probs_gb300 as lp
    with pytest.raises(TypeError):
        lp.read_status(torch.zeros(256, dtype=torch.uint8))
    with pytest.raises(TypeError):
        lp._dev_f32(torch.zeros(4), "temperatures")
    with pytest.raises(TypeError):
        lp._dev_u32(torch.zeros(4, dtype=torch.int32), "tokens")
    with pytest.raises(TypeError):
        lp._dev_u8(torch.zeros(4, dtype=torch.uint8), "echo", 4)


def test_row_kernels_static_shared_memory_keeps_rings_aligned(tmp_path, capfd):
    # The rings live in dynamic shared memory, which starts where a kernel's static shared
    # memory ends: a static size off a multiple of 128 bytes would make every warp's
    # 512-byte copies and 16-byte reads touch five 128-byte rows instead of four.
    from ragged_log_probs_gb300 import _build
    _build.build(force=True, ptxas_verbose=True, out=str(tmp_path / "liblp_check.so"))
    report = capfd.readouterr().err
    sizes, kernel = {}, None
    for line in report.splitlines():
        m = re.search(r"Compiling entry function '(\S+)'", line)
        if m:
            kernel = m.group(1)
            continue
        m = re.search(r"Used \d+ registers.*?(\d+) bytes smem", line)
        if m and kernel and "k_rows" in kernel:
            sizes[kernel] = int(m.group(1))
    assert len(sizes) >= 12, report[-2000:]
    assert all(v % 128 == 0 for v in sizes.values()), sizes
