"""Out-of-bounds write check without a sanitizer: every output and the workspace sit
inside a larger buffer filled with a canary pattern, the C ABI is called with
pointers into the middle, and the guard regions must come back untouched."""
import ctypes

import numpy as np
import pytest

import synth
from lp_util import dev_f32, dev_i32, dev_inputs, part_of

pytestmark = pytest.mark.gpu

CANARY = 0x7FC0DEAD  # a NaN bit pattern no kernel writes
GUARD = 1024         # 4-byte words on each side


@pytest.fixture(scope="module")
def lp():
    from lm_head_linear_tcgen05_gb300 import _build
    _build.build()
    import lm_head_linear_tcgen05_gb300 as mod
    import torch
    assert mod.lp_device_supported()
    torch.cuda.set_device(0)
    return mod


class Guarded:
    """n 4-byte words with GUARD canary words before and after."""

    def __init__(self, n):
        import torch
        self.n = n
        self.buf = torch.full((n + 2 * GUARD,), CANARY, dtype=torch.int32, device="cuda")

    @property
    def ptr(self):
        return self.buf.data_ptr() + 4 * GUARD

    def intact(self):
        b = self.buf.cpu().numpy().view(np.uint32)
        return bool(np.all(b[:GUARD] == CANARY) and np.all(b[GUARD + self.n:] == CANARY))


def test_forward_and_backward_write_only_inside_their_buffers(lp):
    part = synth.ranges_partition(3000, 3072, [0, 1000, 1000, 3072])     # empty and padded shards
    T, H = 137, 200
    inp = synth.forward_inputs(T, H, part, tau=0.7, seed=31, bias_std=0.1)
    X, W, b, y = dev_inputs(inp)
    P = part_of(part)
    L = lp.lib()
    cp, keep = lp._c_partition(P)
    logp, lse, ent = Guarded(T), Guarded(T), Guarded(T)
    ss = Guarded(3 * 3 * T)
    ws_n = lp.lp_workspace_size(lp.LP_OP_FORWARD, T, H, P)
    ws = Guarded((ws_n + 3) // 4)
    out = lp._Outputs(logp.ptr, lse.ptr, ent.ptr, ss.ptr)
    Wp = lp._ptr_array(W)
    bp = lp._ptr_array(b)
    st = L.lp_forward(X.data_ptr(), T, H, Wp, bp, ctypes.byref(cp), y.data_ptr(), inp.tau, ctypes.byref(out),
                      ws.ptr, ws_n, lp._stream(X.device))
    assert st == 0 and lp.lp_get_device_error() == 0
    for gbuf in (logp, lse, ent, ss, ws):
        assert gbuf.intact()

    g = dev_f32(synth.upstream_grad(T, seed=31))
    dX = Guarded(T * H)
    dW = [Guarded((e - s) * H) if e > s else None for s, e in part.ranges]
    db = [Guarded(e - s) if e > s else None for s, e in part.ranges]
    wsb_n = lp.lp_workspace_size(lp.LP_OP_BACKWARD, T, H, P)
    wsb = Guarded((wsb_n + 3) // 4)
    dWp = (ctypes.c_void_p * 3)(*[d.ptr if d else None for d in dW])
    dbp = (ctypes.c_void_p * 3)(*[d.ptr if d else None for d in db])
    lse_t = lse.buf[GUARD:GUARD + T].view(dtype=__import__("torch").float32)
    ent_t = ent.buf[GUARD:GUARD + T].view(dtype=__import__("torch").float32)
    st = L.lp_backward(X.data_ptr(), T, H, Wp, bp, ctypes.byref(cp), y.data_ptr(), inp.tau, lse_t.data_ptr(),
                       g.data_ptr(), ent_t.data_ptr(), g.data_ptr(), dX.ptr, dWp, dbp, wsb.ptr, wsb_n,
                       lp._stream(X.device))
    assert st == 0 and lp.lp_get_device_error() == 0
    for gbuf in [dX, wsb] + [d for d in dW + db if d is not None]:
        assert gbuf.intact()


def test_logits_and_replay_write_only_inside_their_buffers(lp):
    part = synth.ranges_partition(9000, 9000, [0, 4096, 4096, 9000])   # row strides multiples of 8
    T = 45
    L_, yl, tau = synth.logits_inputs(T, part, 0.7, seed=2)
    from lp_util import dev_bf16
    Ld = [dev_bf16(a) if a.shape[1] else None for a in L_]
    P = part_of(part)
    Lb = lp.lib()
    cp, keep = lp._c_partition(P)
    ld = lp._logits_ld(Ld, P, T)
    logp, lse, ent, ss = Guarded(T), Guarded(T), Guarded(T), Guarded(9 * T)
    out = lp._Outputs(logp.ptr, lse.ptr, ent.ptr, ss.ptr)
    st = Lb.lp_forward_from_logits(lp._ptr_array(Ld), ld, T, ctypes.byref(cp), dev_i32(yl).data_ptr(), tau,
                                   ctypes.byref(out), None, 0, lp._stream(Ld[0].device))
    assert st == 0 and lp.lp_get_device_error() == 0
    assert all(x.intact() for x in (logp, lse, ent, ss))

    inp = synth.forward_inputs(T, 64, part, tau=0.7, seed=3)
    X, W, _, _ = dev_inputs(inp)
    ids, yr = synth.replay_ids(T, part, seed=4)
    logp, lse, ss = Guarded(T), Guarded(T), Guarded(9 * T)
    out = lp._Outputs(logp.ptr, lse.ptr, None, ss.ptr)
    st = Lb.lp_top_p_replay(X.data_ptr(), T, 64, lp._ptr_array(W), None, ctypes.byref(cp), dev_i32(ids).data_ptr(),
                            dev_i32(yr).data_ptr(), 0.7, ctypes.byref(out), None, 0, lp._stream(X.device))
    assert st == 0 and lp.lp_get_device_error() == 0
    assert all(x.intact() for x in (logp, lse, ss))
