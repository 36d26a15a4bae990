"""Failure detection on the GPU without a fault: a pipeline wait that runs
out of polls ends the call with KVC_ERR_TIMEOUT, read on the host, and leaves
the context usable.

KVC_OPT_WAIT_LIMIT set to one poll makes the scans' first waits give up (the
first key tile of a CTA takes microseconds to arrive).  A CTA whose wait gave
up stops its pipeline, waits for the copies and MMAs it already issued, and
returns; nothing traps.  With the limit back at its default the next call
must be clean and match the oracle.
"""

import pytest
import torch

from synth import get_config, make_layer_inputs
from tests import kvc_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from attention_score_kv_gb300 import build
    build.build()
    import attention_score_kv_gb300.kvc as kvc
    return kvc


def test_a_wait_that_runs_out_reports_timeout_then_the_next_call_is_clean(K):
    cfg = get_config("tiny", S=4096, C=4096, H_q=8, H_kv=2, D=128, W=32, pool_k=7, K_l=300, recent=32,
                     hh_frac=0.02, seed=70)
    inp = make_layer_inputs(cfg)
    K_l, K_l_ref = U.kl_vector(cfg, K)
    K.kvc_check_status()                                   # start from a clear status word
    K.kvc_set_option(K.KVC_OPT_WAIT_LIMIT, 1)
    try:
        q, k, v = U.to_dev(inp)
        k_out, v_out, pos, off = K.retained_outputs(cfg.B, cfg.H_kv, cfg.S, cfg.D, K_l)
        ws = K.workspace(cfg.B, cfg.H_q, cfg.H_kv, cfg.D, cfg.W, cfg.b_s, max(K_l), cfg.pool_k)
        K.kvc_compress_layer(cfg.N, 0, cfg.B, cfg.S, cfg.C, cfg.H_q, cfg.H_kv, cfg.D, cfg.W, K_l, cfg.sink,
                             cfg.recent, cfg.pool_k, cfg.b_s, q, k, v, k_out, v_out, pos, ws)
        with pytest.raises(K.KvcError) as ei:
            K.kvc_check_status()
        assert ei.value.code == K.KVC_ERR_TIMEOUT
    finally:
        K.kvc_set_option(K.KVC_OPT_WAIT_LIMIT, 0)
    # the status word was read and cleared; the context still works
    k_out, v_out, pos, off = U.run_compress(K, cfg, inp, K_l)
    for h in range(cfg.H_kv):
        o = U.oracle_head(cfg, inp, 0, h)
        U.check_head_outputs(k_out, v_out, pos, off, inp, cfg, 0, h, K_l_ref[h], o["s"], f"after timeout h={h}")
