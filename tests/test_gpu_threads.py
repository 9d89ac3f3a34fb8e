"""Host threads calling the library at once, each on its own stream.

The plan cache, the per-device launch set-up and the device error word are
shared by every caller of the process.  Two threads run the ring forward and
backward of different problems concurrently (bf16 on the tensor cores, float32
on the FFMA kernels) and their results must equal a run of the same problems
from one thread: bit for bit where the kernels fix the summation order (O,
LSE, dK, dV), within the parity bar for dQ (its partials are added into the
float32 accumulator in the order L2 resolves them).
"""

import threading

import pytest
import torch

from tile_attention_lse_gb300 import api

from helpers import TOL_GRAD_REL, make_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"

CASES = [
    # name, batch, seqlen, heads_q, heads_kv, head_dim, cp, dtype
    ("bf16_gqa", 1, 4096, 4, 2, 128, 4, torch.bfloat16),
    ("f32_d64", 2, 1024, 2, 2, 64, 2, torch.float32),
]


def _problem(case):
    _, b, s, H, Hkv, d, cp, dtype = case
    p = api.Problem(batch=b, heads_q=H, heads_kv=Hkv, head_dim=d, cp=cp, seqlen=s, dtype=dtype)
    q, k, v, do = make_inputs(b, s, H, Hkv, d, seed=31, dtype=dtype, with_do=True)
    return p, [x.to(DEV) for x in (q, k, v, do)]


def _run(p, q, k, v, do, reps):
    out = None
    for _ in range(reps):
        o, lse = api.ring_attn_fwd(p, q, k, v)
        dq, dk, dv = api.ring_attn_bwd(p, q, k, v, o, lse, do)
        out = (o, lse, dq, dk, dv)
    return out


def test_two_threads_match_one_thread():
    probs = [_problem(c) for c in CASES]
    results = [None] * len(CASES)
    errors = []
    start = threading.Barrier(len(CASES))

    def worker(i):
        try:
            p, (q, k, v, do) = probs[i]
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                start.wait()
                results[i] = _run(p, q, k, v, do, reps=3)
                stream.synchronize()
        except Exception as e:  # reported on the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(CASES))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    torch.cuda.synchronize()
    assert api.device_error() == 0

    for i, (p, (q, k, v, do)) in enumerate(probs):
        ref = _run(p, q, k, v, do, reps=1)
        torch.cuda.synchronize()
        got = results[i]
        for name, a, r in zip(("O", "LSE", "dK", "dV"), (got[0], got[1], got[3], got[4]),
                              (ref[0], ref[1], ref[3], ref[4])):
            assert torch.equal(a, r), (CASES[i][0], name)
        scale = float(ref[2].float().abs().max())
        assert float((got[2].float() - ref[2].float()).abs().max()) <= TOL_GRAD_REL * scale, CASES[i][0]
