"""CPU checks of the forward kernel's synchronisation protocols on the executable model in
pipeline_model.py: two Q tiles with a dedicated S-issuer warp, at d = 64 (three rotating S
buffers) and at d = 128, bf16 and e4m3 (one S buffer both Q tiles share, P in a tensor-memory
area per tile).

The protocols as built pass random schedules, with K/V copies landing in any order. The other
checks show each model failing when one piece of its protocol is removed, so the passing runs
mean something.
"""
from pipeline_model import sweep


def test_protocol_as_built_passes_random_schedules():
    assert sweep(400, case_seed=1, M=3) is None
    assert sweep(400, case_seed=2, M=3) is None


def test_two_barriers_per_tile_break_the_phase_window():
    # With S issued by another warp a tile can have three S products outstanding; two barriers
    # per tile then let a parity wait see its barrier two phases away.
    failure = sweep(400, case_seed=1, M=2)
    assert failure is not None and "phase window" in failure


def test_missing_buffer_free_wait_is_caught():
    failure = sweep(100, case_seed=3, M=3, skip_s_free=True)
    assert failure is not None and "overwrites buffer" in failure


def test_missing_rescale_wait_is_caught():
    failure = sweep(100, case_seed=4, M=3, skip_rescale_wait=True)
    assert failure is not None and "rescaled" in failure


def test_shared_s_protocol_as_built_passes_random_schedules():
    # d = 128 bf16: four K/V stages (the even count below five that shared memory holds)
    assert sweep(400, case_seed=21, mode="s1", ns=4) is None
    assert sweep(400, case_seed=25, mode="s1", ns=4) is None


def test_odd_ring_breaks_the_phase_window():
    # Five stages put K and V tiles in turn through each stage; a PV issuer whose tile has no keys
    # in a work tile then passes a V stage two phases early. The kernel keeps the count even.
    failure = sweep(400, case_seed=21, mode="s1", ns=5)
    assert failure is not None and "phase window" in failure
    failure = sweep(400, case_seed=24, M=3, ns=5)
    assert failure is not None and "phase window" in failure


def test_shared_s_missing_load_wait_is_caught():
    # the next S may enter the shared buffer only once the softmax owning the last one loaded it
    failure = sweep(100, case_seed=13, mode="s1", ns=4, skip_s_free=True)
    assert failure is not None and "before the softmax loaded it" in failure


def test_shared_s_missing_pv_wait_is_caught():
    # P_j overwrites the tile's P area only after PV_{j-1} has read it
    failure = sweep(100, case_seed=14, mode="s1", ns=4, skip_rescale_wait=True)
    assert failure is not None and "before the PV before it read P" in failure
