"""CPU-side checks of the C ABI: the library builds and loads, exports every entry point the
header declares, its ctypes mirrors match the C struct layouts, and invalid arguments are
rejected before any device work (no GPU needed)."""
import ctypes as C
import os
import re
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dgcanvas.h")


@pytest.fixture(scope="module")
def dg():
    from uniform_state_denoising_vocab_b300 import build
    build.build()
    import uniform_state_denoising_vocab_b300 as m
    m.lib()
    return m


def _declared():
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"DG_API\s+[\w\s\*]+?\b(dg_\w+)\s*\(", txt)))


def test_exports_every_declared_symbol(dg):
    names = _declared()
    assert {"dg_canvas_stats", "dg_canvas_step", "dg_canvas_loop", "dg_workspace_bytes"} <= set(names)
    out = subprocess.run(["nm", "-D", "--defined-only", str(dg._LIB_PATH)], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(dg_\w+)$", out, re.M))
    for n in names:
        assert n in exported, n
        assert hasattr(dg.lib(), n)


def test_struct_layouts_match_header(dg):
    prog = r"""
#include <stdio.h>
#include <stddef.h>
#include "dgcanvas.h"
#define P(T, f) printf(#T "." #f " %zu\n", offsetof(T, f));
int main(void) {
  printf("dg_head_desc %zu\n", sizeof(dg_head_desc));
  P(dg_head_desc, h) P(dg_head_desc, h_scale) P(dg_head_desc, w) P(dg_head_desc, w_scale)
  P(dg_head_desc, inv_temp) P(dg_head_desc, h_block_scale) P(dg_head_desc, w_block_scale)
  printf("dg_canvas_state %zu\n", sizeof(dg_canvas_state));
  printf("dg_stop_rule %zu\n", sizeof(dg_stop_rule));
  printf("dg_loop_params %zu\n", sizeof(dg_loop_params));
  P(dg_loop_params, keep_sched) P(dg_loop_params, seed) P(dg_loop_params, start_pass)
  P(dg_loop_params, trace_h) P(dg_loop_params, trace_entropy) P(dg_loop_params, trace_timeline)
  P(dg_loop_params, temp_start) P(dg_loop_params, temp_end) P(dg_loop_params, row_offset)
  P(dg_loop_params, trace_sm_clock)
  P(dg_stop_rule, keep_rule) P(dg_stop_rule, redraw_mode) P(dg_stop_rule, mask_id)
  printf("dg_synth_params %zu\n", sizeof(dg_synth_params));
  P(dg_synth_params, n_content) P(dg_synth_params, s_pad) P(dg_synth_params, status)
  return 0;
}
"""
    with tempfile.TemporaryDirectory() as t:
        src = os.path.join(t, "layout.c")
        exe = os.path.join(t, "layout")
        open(src, "w").write(prog)
        subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), src, "-o", exe], check=True)
        lines = subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split("\n")
    got = dict(l.split() for l in lines if l.strip())
    m = {"dg_head_desc": dg.HeadDesc, "dg_canvas_state": dg.CanvasState,
         "dg_stop_rule": dg.StopRule, "dg_loop_params": dg.LoopParams,
         "dg_synth_params": dg.SynthParams}
    for k, v in got.items():
        if "." in k:
            t, f = k.split(".")
            assert getattr(m[t], f).offset == int(v), k
        else:
            assert C.sizeof(m[k]) == int(v), k


def _desc(dg, **kw):
    d = dict(B=1, S=256, d=64, V=4096, h_dtype=dg.DG_BF16, w_dtype=dg.DG_BF16, h=4096, h_scale=None,
             w=8192, w_scale=None, inv_temp=1.0)
    d.update(kw)
    return dg.HeadDesc(**d)


@pytest.mark.parametrize("kw,code", [
    (dict(B=0), -1), (dict(S=0), -1), (dict(V=0), -1), (dict(d=0), -1), (dict(S=2048), -3),
    (dict(inv_temp=0.0), -1), (dict(inv_temp=-1.0), -1), (dict(w=None), -1),
    (dict(h_dtype=2, w_dtype=1), -3), (dict(h_dtype=0, w_dtype=1), -3),
    (dict(w_dtype=2), -1),                      # e4m3 head without scales
    (dict(d=60), -2),                           # 60 * 2 bytes is not a multiple of 16
    (dict(w=8200), -2),                         # misaligned pointer
])
def test_invalid_arguments_rejected_without_device(dg, kw, code):
    desc = _desc(dg, **kw)
    n = C.c_size_t(0)
    assert dg.lib().dg_workspace_bytes(C.byref(desc), C.byref(n)) == code
    assert dg.lib().dg_workspace_bytes(None, C.byref(n)) == -1


def test_step_argument_checks(dg):
    desc = _desc(dg)
    L = dg.lib()
    # null canvases and negative keep are rejected before any device query
    assert L.dg_canvas_step(C.byref(desc), None, None, 1, 0, 0, None, None, None, None, None, None,
                            None, None, 0, None, None) == -1
    assert L.dg_canvas_step(C.byref(desc), 16, 16, -1, 0, 0, None, None, None, None, None, None,
                            None, None, 0, None, None) == -1
    # a state without a stop rule is rejected
    assert L.dg_canvas_step(C.byref(desc), 16, 16, 1, 0, 0, None, None, None, None, None, 32,
                            None, None, 0, None, None) == -1


def test_host_step_argument_checks(dg):
    """dg_canvas_step_host rejects missing buffers and bad descriptors before any device work."""
    desc = _desc(dg)
    L = dg.lib()
    n = C.c_size_t(0)
    assert L.dg_workspace_bytes_host(None, C.byref(n)) == -1
    assert L.dg_workspace_bytes_host(C.byref(desc), None) == -1
    assert L.dg_workspace_bytes_host(C.byref(_desc(dg, B=0)), C.byref(n)) == -1
    assert L.dg_workspace_bytes_host(C.byref(_desc(dg, w=8200)), C.byref(n)) == -2
    # null canvases, null h or null workspace
    assert L.dg_canvas_step_host(C.byref(desc), None, 16, None, 1, 0, 0, None, None, 256, 1 << 20,
                                 None, None) == -1
    assert L.dg_canvas_step_host(C.byref(desc), 16, None, None, 1, 0, 0, None, None, 256, 1 << 20,
                                 None, None) == -1
    assert L.dg_canvas_step_host(C.byref(_desc(dg, h=None)), 16, 16, None, 1, 0, 0, None, None,
                                 256, 1 << 20, None, None) == -1
    assert L.dg_canvas_step_host(C.byref(desc), 16, 16, None, 1, 0, 0, None, None, None, 1 << 20,
                                 None, None) == -1


def test_selftest_rejects_null_status(dg):
    assert dg.lib().dg_selftest_wait_timeout(None, None) == -1


def test_quantise_e4m3_argument_checks(dg):
    L = dg.lib()
    assert L.dg_quantize_e4m3(None, 4, 16, 16, 16, None, None) == -1      # no input
    assert L.dg_quantize_e4m3(16, 4, 16, None, 16, None, None) == -1      # no codes
    assert L.dg_quantize_e4m3(16, 0, 16, 16, 16, None, None) == -1        # no rows
    assert L.dg_quantize_e4m3(16, 4, 0, 16, 16, None, None) == -1         # no width
    assert L.dg_quantize_e4m3(17, 4, 16, 16, 16, None, None) == -2        # misaligned input


def test_status_strings(dg):
    for code in (0, -1, -2, -3, -4, -5, 1, 2, 4):
        s = dg.dg_status_string(code)
        assert s and "unknown" not in s
    assert dg.lib().dg_version() >= 100


def test_rule_and_schedule_checks(dg):
    """Keep / re-draw variants and the temperature schedule are validated before any device
    work: an unknown keep rule or re-draw mode, a mask id outside [0, V), a negative or
    one-sided temperature schedule are DG_ERR_INVALID_ARG."""
    desc = _desc(dg)
    L = dg.lib()
    bad = [dg.pass_rule(keep_rule=2), dg.pass_rule(mask_id=4096), dg.pass_rule(mask_id=-1)]
    bad[2].redraw_mode = dg.REDRAW_MASK
    r3 = dg.pass_rule()
    r3.redraw_mode = 5
    bad.append(r3)
    for rule in bad:
        assert L.dg_canvas_step(C.byref(desc), 16, 16, 1, 0, 0, None, None, None, None, None,
                                None, C.byref(rule), None, 0, None, None) == -1
    for ts, te in ((-1.0, 0.4), (0.8, 0.0), (0.8, -0.4), (float("nan"), 0.4)):
        params = dg.LoopParams(rule=dg.pass_rule(), keep_k0=1, temp_start=ts, temp_end=te)
        params.rule.max_passes = 4
        params.rule.stable_passes = 2
        desc_h = _desc(dg, h=8192)
        assert L.dg_canvas_loop(C.byref(desc_h), 16, 8192, C.byref(params), 16, None, 32, None,
                                None, None, None, 0, None, None) == -1
