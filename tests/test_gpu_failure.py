"""Failure detection on the GPU without a GPU fault: a test hook makes the operand
producer leave one pipeline stage unarmed, so the MMA issuer's bounded wait runs out.
The kernel must record FG_ERR_DEVICE_TIMEOUT in the status word, every role must exit
cleanly (no trap, no hang), and the context must stay usable for the next call."""
import pytest

import cases as C

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def fg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import moe_fp8_e4m3_gb300 as lib
    return lib


def test_stalled_pipeline_times_out_and_context_survives(fg):
    from gpu_util import GuardedOut, dev
    case = C.dense_case(41, 256, 512, 512, False, "bf16")
    args = [dev(case[k]) for k in ("a", "sfa", "b", "sfb")]
    out = GuardedOut(256, 512, "bf16")
    assert fg.get_device_error()[0] == 0
    fg.debug_inject_stall(True, 200_000)         # 200 ms per wait
    try:
        fg.fp8_gemm_nt(*args, out.tensor)        # the launch itself succeeds
        st, detail = fg.get_device_error()
    finally:
        fg.debug_inject_stall(False)
    assert st == fg.FG_ERR_DEVICE_TIMEOUT, (st, hex(detail))
    assert detail & 0x200
    out.check_guards()
    # the same call, now without the stall, on the same context
    fg.fp8_gemm_nt(*args, out.tensor)
    assert fg.get_device_error()[0] == 0
    C.compare(out.values(), C.dense_ref(case), "after time-out")


@pytest.mark.parametrize("split", ["1", "2"])
def test_fp4_stalled_pipeline_times_out_and_context_survives(fg, split, monkeypatch):
    """The FP8 x FP4 GEMM's bounded waits: with the operand producer holding back its first
    stage (host-side stall hook), the call records a time-out and returns; the same call
    then runs correctly on the same context (one CTA per tile and split-K clusters)."""
    from gpu_util import GuardedOut, dev
    monkeypatch.setenv("FG_FORCE_SPLIT", split)
    case = C.fp4_dense_case(42, 64, 512, 1024, True, "f32")
    args = [dev(case[k]) for k in ("a", "sfa", "b", "sfb")]
    c_t = dev(case["c"])
    out = GuardedOut(64, 512, "f32")
    assert fg.get_device_error()[0] == 0
    fg.debug_inject_stall(True, 200_000)
    try:
        fg.fp8_fp4_gemm_nt(*args, out.tensor, c=c_t)
        st, detail = fg.get_device_error()
    finally:
        fg.debug_inject_stall(False)
    assert st == fg.FG_ERR_DEVICE_TIMEOUT, (st, hex(detail))
    assert detail & 0x200
    out.check_guards()
    fg.fp8_fp4_gemm_nt(*args, out.tensor, c=c_t)
    assert fg.get_device_error()[0] == 0
    C.compare(out.values(), C.fp4_dense_ref(case), "fp4 after time-out")
