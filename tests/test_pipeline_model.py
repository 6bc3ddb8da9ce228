"""CPU checks of the forward kernel's synchronisation protocols on the executable models in
pipeline_model.py: d = 64 (three rotating S buffers, a dedicated S-issuer warp) and e4m3 with P
in shared memory.

Both protocols as built (d = 64 with three barriers per Q tile) pass random schedules. The
other checks show each model failing when one piece of its protocol is removed, so the passing
runs mean something.
"""
from pipeline_model import sweep, sweep_psmem


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


def test_psmem_protocol_as_built_passes_random_schedules():
    assert sweep_psmem(400, case_seed=5) is None


def test_psmem_missing_read_wait_is_caught():
    # S_{j+1} must wait until the softmax has loaded S_j from the tile's one TMEM buffer
    failure = sweep_psmem(100, case_seed=6, skip_read_wait=True)
    assert failure is not None and "before the softmax loaded it" in failure


def test_psmem_missing_pv_wait_is_caught():
    # P_j must wait for PV_{j-1}, which reads the same shared-memory P tile (and O for rescales)
    failure = sweep_psmem(100, case_seed=7, skip_pv_wait=True)
    assert failure is not None and ("before its PV read it" in failure or "rescaled" in failure)
