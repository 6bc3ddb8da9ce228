"""CPU checks of the d = 64 forward kernel's synchronisation protocol (three rotating S buffers,
a dedicated S-issuer warp), on the executable model in pipeline_model.py.

The protocol as built (three barriers per Q tile) passes random schedules. Each check below it
shows the model failing when one piece of the protocol is removed, so the passing run means
something.
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
