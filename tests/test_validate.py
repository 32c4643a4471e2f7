"""echo_pool_validate / echo_pool_validate_host: the metadata invariants of one pool
(ECHO review, section 5.1 metadata table: the five arrays describe one bijection between
occupied slots and resident host rows; section 5.2 "Free": a freed slot has free = 1,
priority = -1 and no map entries).

The host form runs here without a GPU: consistent pools from the workload generator
pass, and each kind of corruption made on the host raises the status bit and counts
in the right field.  The device form is checked on corrupted metadata uploaded from
the host, and on the pools a long replayed run leaves (tests/test_gpu_multistep.py)."""
import numpy as np
import pytest
import torch

import sparse_attention_kv_fp8_gb300 as echo
from sparse_attention_kv_fp8_gb300 import _build
from sparse_attention_kv_fp8_gb300 import workload as wl

INF = echo.INF


@pytest.fixture(scope="module", autouse=True)
def lib():
    _build.build()
    return echo.load_library()


def _state(n_g=300, n_h=2000, n_res=250, seed=3):
    rows = wl.random_resident_rows(n_h, n_res, seed)
    st = wl.resident_pool(n_g, n_h, rows, wl.random_clocks(n_res, 50, seed), seed)
    return dict(free=st.gpu_token_free.copy(), prio=st.gpu_token_priority.copy(),
                to_host=st.gpu_token_to_host.copy(), host_to_gpu=st.host_token_to_gpu.copy(), n_free=int(st.n_free))


def _check(m, reserve=None):
    return echo.echo_pool_validate_host(m["free"], m["prio"], m["to_host"], m["host_to_gpu"], m["n_free"],
                                        reserve=reserve)


def test_consistent_pools_pass():
    for n_res in (0, 120, 300):
        bad, rep = _check(_state(n_res=n_res))
        assert not bad, rep
        assert rep["occupied"] == n_res and rep["free"] == 300 - n_res and rep["resident"] == n_res
        assert rep["slot_state"] == rep["slot_map"] == rep["row_map"] == rep["counter"] == rep["reserve"] == 0


def _occupied_slot(m):
    return int(np.nonzero(m["free"] == 0)[0][0])


def _free_slot(m):
    return int(np.nonzero(m["free"] == 1)[0][0])


@pytest.mark.parametrize("kind,field", [
    ("to_host_elsewhere", "slot_map"),     # an occupied slot names a host row that maps to another slot
    ("row_map_elsewhere", "row_map"),      # a resident row names a slot that holds another row
    ("row_map_out_of_range", "row_map"),
    ("claim_mark_left", "row_map"),        # a recall's claim mark (negative) left in the map
    ("free_with_priority", "slot_state"),  # free = 1 but a priority
    ("free_with_row", "slot_state"),       # free = 1 but a host row
    ("occupied_without_row", "slot_state"),
    ("bad_free_flag", "slot_state"),
    ("counter_off", "counter"),
])
def test_each_corruption_is_seen(kind, field):
    m = _state()
    s, f = _occupied_slot(m), _free_slot(m)
    h = int(m["to_host"][s])
    if kind == "to_host_elsewhere":
        other = int(np.nonzero((m["free"] == 0) & (np.arange(m["free"].size) != s))[0][0])
        m["to_host"][s] = m["to_host"][other]
    elif kind == "row_map_elsewhere":
        m["host_to_gpu"][h] = f
    elif kind == "row_map_out_of_range":
        m["host_to_gpu"][int(np.nonzero(m["host_to_gpu"] == INF)[0][0])] = m["free"].size + 5
    elif kind == "claim_mark_left":
        m["host_to_gpu"][int(np.nonzero(m["host_to_gpu"] == INF)[0][0])] = -(2**31) + 7
    elif kind == "free_with_priority":
        m["prio"][f] = 3
    elif kind == "free_with_row":
        m["to_host"][f] = 17
    elif kind == "occupied_without_row":
        m["host_to_gpu"][h] = INF
        m["to_host"][s] = INF
    elif kind == "bad_free_flag":
        m["free"][s] = 2
    elif kind == "counter_off":
        m["n_free"] += 1
    bad, rep = _check(m)
    assert bad, (kind, rep)
    assert rep[field] >= 1, (kind, rep)


def test_reserve_checks():
    m = _state(n_res=200)
    fs = np.nonzero(m["free"] == 1)[0][:5]
    m["free"][fs] = 0
    m["prio"][fs] = -2            # reserved: not free, priority -2, no row
    m["n_free"] -= 5
    bad, rep = _check(m, reserve=fs)
    assert not bad and rep["reserved"] == 5, rep
    bad, rep = _check(m, reserve=fs[:4])          # a reserved slot the reserve does not list
    assert bad and rep["reserve"] == 1
    listed = fs.copy()
    listed[2] = int(np.nonzero(m["prio"] >= 0)[0][0])   # the reserve lists an occupied slot
    bad, rep = _check(m, reserve=listed)
    assert bad and rep["reserve"] >= 1
    listed = fs.copy()
    listed[2] = fs[3]                             # one reserved slot twice, another left out
    bad, rep = _check(m, reserve=listed)
    assert bad and rep["reserve"] == 1 and rep["reserve_balance"] == int(fs[2] - fs[3])
    m["to_host"][fs[0]] = 11                      # a reserved slot with a host row
    bad, rep = _check(m, reserve=fs)
    assert bad and rep["slot_state"] == 1


def test_prefetched_mark_is_an_occupied_slot():
    m = _state()
    m["prio"][_occupied_slot(m)] = -3             # filled by the direct-to-slot prefetch this step
    bad, rep = _check(m)
    assert not bad, rep


def test_bad_arguments_are_rejected(lib):
    assert lib.echo_pool_validate_host(None, None, 0, None) == -echo.ECHO_EINVAL


@pytest.mark.gpu
def test_device_validate_sees_corruption_made_on_the_host():
    m = _state(n_g=5000, n_h=40000, n_res=4500, seed=5)
    host = torch.zeros((40000, echo.KV_ELEMS), dtype=torch.int16, pin_memory=True)
    pool = echo.Pool(5000, host)
    report = torch.zeros(len(echo.VAL_FIELDS), dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def load(mm):
        pool.free.copy_(torch.from_numpy(mm["free"]))
        pool.prio.copy_(torch.from_numpy(mm["prio"]))
        pool.to_host.copy_(torch.from_numpy(mm["to_host"]))
        pool.host_to_gpu.copy_(torch.from_numpy(mm["host_to_gpu"]))
        pool.counters.copy_(torch.tensor([mm["n_free"], 0, 0, 0], dtype=torch.int32))

    load(m)
    echo.echo_pool_validate(pool, report, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    dev_rep = dict(zip(echo.VAL_FIELDS, report.cpu().tolist()))
    assert dev_rep == _check(m)[1]
    s = _occupied_slot(m)
    m["host_to_gpu"][int(m["to_host"][s])] = _free_slot(m)
    m["n_free"] -= 1
    load(m)
    echo.echo_pool_validate(pool, report, status)
    torch.cuda.synchronize()
    assert int(status.item()) & echo.DEV_INVARIANT
    dev_rep = dict(zip(echo.VAL_FIELDS, report.cpu().tolist()))
    assert dev_rep == _check(m)[1] and dev_rep["row_map"] >= 1 and dev_rep["counter"] == 1
