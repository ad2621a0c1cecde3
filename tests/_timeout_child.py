"""Child process of test_gpu_timeout.py (not a test module): runs the test-hook
build of the library, whose switch makes pass 1's bounded wait for the in-launch
K/V quantizer poll a word that nothing sets.  Prints one JSON line."""
import ctypes
import json
import os
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import mixed_precision_attention_gb300._lib as L  # noqa: E402

L.LIB_PATH = sys.argv[1]

import numpy as np  # noqa: E402
import torch  # noqa: E402

import mixed_precision_attention_gb300 as apa  # noqa: E402
import oracle  # noqa: E402
from mixed_precision_attention_gb300 import synth  # noqa: E402

lib = L.load()
lib.apa_test_stuck_quantizer_flags.argtypes = [ctypes.c_int]
lib.apa_test_stuck_quantizer_flags.restype = ctypes.c_int
# one KV head: a single pass-1 CTA, so the K/V tiles are quantized inside its launch
w = synth.small(B=1, Hq=2, Hkv=1, Nq=128, Nkv=4096, d=64, sink_gain=4.0, n_outliers=2, seed=9)
q, k, v = synth.generate(w)
tq, tk, tv = (synth.to_torch_bf16(a, "cuda") for a in (q, k, v))
stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def call():
    t0 = time.time()
    out, _, _ = apa.attention(tq, tk, tv, causal=True, eps=0.005)
    st = lib.apa_check_error(stream)  # synchronizes; the device error word, cleared
    return out, st, time.time() - t0


call()  # warm: module load, workspace
lib.apa_test_stuck_quantizer_flags(1)
_, stuck_status, stuck_s = call()
lib.apa_test_stuck_quantizer_flags(0)
out, after_status, _ = call()
got = out.cpu().numpy().astype(np.float64)
ref = oracle.apa(q, k, v, eps=0.005)["out"]
print(json.dumps(dict(stuck_status=stuck_status, stuck_seconds=stuck_s, after_status=after_status,
                      after_max_err=float(np.abs(got - ref).max()), after_finite=bool(np.isfinite(got).all()))))
