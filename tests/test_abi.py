"""The C-ABI library loads, exports every symbol include/cp.h declares, and its
host-side schedule checker works -- no GPU needed, no compute calls."""
import ctypes
import os
import re

import pytest

import synth
from persistent_megakernel_streaming_gb300 import build, cp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build.build()
    return cp.lib()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "cp.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(cp_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for n in ("cp_create", "cp_frame", "cp_frame_split", "cp_debug_logits", "cp_status", "cp_destroy",
              "cp_strerror"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for n in declared_symbols():
        assert hasattr(L, n), n
    assert sorted(cp.EXPORTS) == declared_symbols()


def test_strerror(L):
    assert L.cp_strerror(0) == b"ok"
    assert b"timed out" in L.cp_strerror(5)


@pytest.mark.parametrize("name,grid,cluster", [("tiny", 16, 4), ("tiny", 148, 4), ("full", 148, 4),
                                               ("full", 152, 4), ("full", 148, 2), ("full", 144, 8),
                                               ("wide", 148, 4), ("full", 8, 4)])
@pytest.mark.parametrize("chunked", [False, True])
def test_schedule_checks_out(L, name, grid, cluster, chunked):
    s = synth.shape(name)
    code, st = cp.plan_check(s, grid, cluster, chunk_waits=chunked)
    assert code == 0, st.message
    assert st.phases == (432 if name != "tiny" else 28)
    # every projection weight byte is streamed exactly once per use
    assert st.weight_bytes == synth.weight_bytes_per_frame(s)
    assert st.min_cta_weight_bytes > 0


@pytest.mark.parametrize("chunked", [False, True])
@pytest.mark.parametrize("corrupt", [1, 2, 3])
def test_checker_catches_broken_schedules(L, corrupt, chunked):
    code, st = cp.plan_check(synth.shape("tiny"), 16, 4, corrupt, chunk_waits=chunked)
    assert code == cp.CP_ERR_PLAN
    assert st.message and st.message != b"ok"


def test_checker_rejects_unsupported_shapes(L):
    s = synth.shape("full")
    s["head_dim"] = 96
    assert cp.plan_check(s, 148, 4)[0] == 2
    s = synth.shape("full")
    s["positions"] = 17
    assert cp.plan_check(s, 148, 4)[0] == 2
    s = synth.shape("full")
    assert cp.plan_check(s, 148, 3)[0] == 1


def test_two_tile_tasks_appear_when_tiles_outnumber_clusters(L):
    # 36 clusters of 4 hold every phase in one round; 16 clusters (64 CTAs) pair
    # tiles where a phase has up to twice as many tiles as clusters
    code, st = cp.plan_check(synth.shape("full"), 144, 4)
    assert code == 0
    one_round = st.tasks
    code, st2 = cp.plan_check(synth.shape("full"), 64, 4)
    assert code == 0, st2.message
    assert st2.weight_bytes == st.weight_bytes


@pytest.mark.parametrize("grid", [148, 144, 64, 16])
@pytest.mark.parametrize("chunked", [False, True])
def test_schedule_for_128_rows_checks_out(L, grid, chunked):
    """A 128-row handle: twice the attention and draw tasks, no two-tile
    projection tasks (its partial-sum exchange has one receive slot), the
    same weight bytes."""
    s = synth.shape("full_r128")
    code, st = cp.plan_check(s, grid, 4, chunk_waits=chunked)
    assert code == 0, st.message
    assert st.phases == 432
    assert st.weight_bytes == synth.weight_bytes_per_frame(s)
    s64 = synth.shape("full")
    code, st64 = cp.plan_check(s64, grid, 4)
    assert code == 0
    # 16 row blocks per kv group instead of 8, 128 draw and first-embedding tasks instead of 64
    assert st.tasks - st64.tasks >= 80 * 8 * 8 + 15 * 64 + 64


def test_max_rows_above_128_is_refused(L):
    s = synth.shape("full")
    s["max_rows"] = 129
    assert cp.plan_check(s, 148, 4)[0] == 2
