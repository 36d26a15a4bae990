"""kvc_compress_layer_deferred_v: the values are uploaded on another stream
while the scans run; only the gather waits on the caller's event.  The
outputs must be bit-identical to kvc_compress_layer's on the same inputs."""

import pytest
import torch

from synth import get_config, make_layer_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import attention_score_kv_gb300.kvc as K
    return K


def _args(cfg):
    return (cfg.N, 0, cfg.B, cfg.S, cfg.C, cfg.H_q, cfg.H_kv, cfg.D, cfg.W)


@pytest.mark.parametrize("with_event", [True, False])
def test_deferred_v_equals_compress_layer(K, with_event):
    cfg = get_config("llama8k")
    inp = make_layer_inputs(cfg, 0)
    dev = "cuda"
    K_l = [cfg.K_l] * cfg.H_kv
    q, k, v = inp.q_win.to(dev), inp.k.to(dev), inp.v.to(dev)
    ws = K.workspace(cfg.B, cfg.H_q, cfg.H_kv, cfg.D, cfg.W, cfg.b_s, max(K_l), cfg.pool_k, device=dev)
    ref = K.retained_outputs(cfg.B, cfg.H_kv, cfg.S, cfg.D, K_l, device=dev)
    K.kvc_compress_layer(*_args(cfg), K_l, cfg.sink, cfg.recent, cfg.pool_k, cfg.b_s, q, k, v,
                         ref[0], ref[1], ref[2], ws)
    got = K.retained_outputs(cfg.B, cfg.H_kv, cfg.S, cfg.D, K_l, device=dev)
    v_late = torch.zeros_like(v)
    v_host = inp.v.contiguous().pin_memory()
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    ev = torch.cuda.Event()
    side.wait_stream(main)           # v_late's zero fill is done before the upload
    with torch.cuda.stream(side):
        v_late.copy_(v_host, non_blocking=True)
        ev.record(side)
    if not with_event:
        main.wait_event(ev)          # no event passed: the values are complete in stream order
    K.kvc_compress_layer_deferred_v(*_args(cfg), K_l, cfg.sink, cfg.recent, cfg.pool_k, cfg.b_s, q, k, v_late,
                                    got[0], got[1], got[2], ws, ev if with_event else None)
    torch.cuda.synchronize()
    K.kvc_check_status()
    for a, b in zip(ref[:3], got[:3]):
        assert torch.equal(a.view(torch.uint8) if a.dtype != torch.int32 else a,
                           b.view(torch.uint8) if b.dtype != torch.int32 else b)
