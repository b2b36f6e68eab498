"""Source rules for the kernels' launch path (no GPU needed).

run() launches with programmatic stream serialisation, so a kernel launched
through it may be scheduled while the previous kernel in the stream is still
running.  Such a kernel must wait for its predecessor before it touches
memory: its first statement is pdl_enter().  A kernel that forgot it would
race with the kernel before it, so this is checked on the sources.
"""
import pathlib
import re

CSRC = pathlib.Path(__file__).resolve().parents[1] / "zero_partitioned_mixed_gb300" / "csrc"
LAUNCH = re.compile(r"\brun(?:_chunked(?:_u)?)?(?:<[^>(]*>)?\(\s*(k_\w+)")
KERNEL = re.compile(r"__global__ void (?:__launch_bounds__\([^)]*\) )?(k_\w+)\(([^)]*)\)\s*\{\n\s*([^\n]*)")


def _sources():
    return {p.name: p.read_text() for p in sorted(CSRC.glob("*.cu")) + sorted(CSRC.glob("*.cuh"))}


def test_kernels_launched_through_run_wait_for_their_predecessor():
    src = _sources()
    launched = {m.group(1) for t in src.values() for m in LAUNCH.finditer(t)}
    first = {}
    for t in src.values():
        for m in KERNEL.finditer(t):
            first.setdefault(m.group(1), []).append(m.group(3).strip())
    # the step, two-pass, fix-up, rollback, gather, reduce-scatter and ZeRO++ kernels
    assert {"k_step_spec", "k_gather", "k_rs", "k_fixup", "k_gather_q8", "k_rs_q"} <= launched
    for k in sorted(launched):
        assert k in first, f"{k} is launched through run() but its definition was not found"
        assert all(f == "pdl_enter();" for f in first[k]), f"{k} does not begin with pdl_enter(): {first[k]}"


def test_run_is_the_only_launch_with_the_attribute():
    # the attribute is set in one place; kernels launched with <<<>>> are plain
    src = _sources()
    hits = [n for n, t in src.items() if "cudaLaunchAttributeProgrammaticStreamSerialization" in t]
    assert hits == ["zero_device.cuh"]
