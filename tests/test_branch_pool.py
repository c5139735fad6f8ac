"""The host branch pool (HPD-Parsing part 2: content branches forked from a shared prefix, reference-
counted release): bookkeeping only, so every test here runs without a GPU."""
import threading

import pytest

import kv_cache_token_fx_gb300 as fx


@pytest.fixture(scope="module")
def lib():
    try:
        return fx.load_library()
    except fx.FxError:
        pytest.skip("library not built")


def test_fork_positions_slots_and_refcount(lib):
    p = fx.BranchPool(prefix_cap=1000, max_branches=3, slot_rows=16)
    assert p.prefix_refs() == 1                 # the parent
    assert p.extend_prefix(100) == 0
    a = p.fork()                                # forks see the prefix as it is at the fork
    assert p.extend_prefix(50) == 100
    b = p.fork()
    assert (a, b) == (0, 1) and p.prefix_refs() == 3
    assert p.append(a, 10) == 0 and p.append(a, 5) == 10 and p.append(b, 3) == 16
    ids, start, length, fork = p.batch()
    assert ids.tolist() == [0, 1] and start.tolist() == [0, 16]
    assert length.tolist() == [15, 3] and fork.tolist() == [100, 150]
    assert p.release(a) == 2                    # parent + b
    c = p.fork()                                # the freed slot is reused, empty, at the new position
    assert c == 0
    ids, start, length, fork = p.batch()
    assert length.tolist() == [0, 3] and fork.tolist() == [150, 150]
    assert p.release_parent() == 2              # children still hold the prefix
    with pytest.raises(fx.FxError):
        p.extend_prefix(1)                      # no growth once the parent is done
    with pytest.raises(fx.FxError):
        p.fork()
    assert p.release(b) == 1 and p.release(c) == 0   # last child: the prefix may be freed


def test_capacity_and_bad_arguments(lib):
    p = fx.BranchPool(prefix_cap=10, max_branches=2, slot_rows=4)
    with pytest.raises(fx.FxError):
        p.extend_prefix(11)
    p.fork()
    p.fork()
    with pytest.raises(fx.FxError):
        p.fork()                                # every slot taken
    assert p.append(1, 4) == 4
    with pytest.raises(fx.FxError):
        p.append(1, 1)                          # slot full
    with pytest.raises(fx.FxError):
        p.append(5, 1)                          # no such branch
    p.release(0)
    with pytest.raises(fx.FxError):
        p.release(0)                            # released twice
    with pytest.raises(fx.FxError):
        fx.BranchPool(prefix_cap=-1, max_branches=1, slot_rows=1)


def test_concurrent_forks_get_distinct_slots(lib):
    p = fx.BranchPool(prefix_cap=0, max_branches=64, slot_rows=8)
    got, lock = [], threading.Lock()

    def worker():
        for _ in range(8):
            s = p.fork()
            with lock:
                got.append(s)

    threads = [threading.Thread(target=worker) for _ in range(8)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert sorted(got) == list(range(64))
    assert p.prefix_refs() == 65
