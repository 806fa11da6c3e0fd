"""Child process of the failure-detection test (run as a script, not collected by pytest).

With a device wait limit of 300 ms (ATTN_WAIT_LIMIT_MS, read when the library makes its first
call), it runs the deterministic backward's main kernel on a workspace whose bytes are all
0xFF and without the prepare step that would zero it: every per-tile turn counter then reads -1,
so the turn every key tile waits for never comes.  The wait must run out, the call must be
reported as ATTN_ERR_TIMEOUT, and the same context must then compute a correct backward.
Prints one JSON line with what it saw."""
import json
import os
import sys
import time

os.environ["ATTN_WAIT_LIMIT_MS"] = "300"
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def main():
    import numpy as np
    import torch

    import oracle
    from exact_attention_50_gb300 import _lib, build
    from exact_attention_50_gb300 import attention as A
    from exact_attention_50_gb300 import workloads as W

    build.build()
    lib = _lib.load()
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream().cuda_stream
    B, Hq, Hkv, N, d = 1, 2, 1, 256, 64
    q, k, v, dout = W.dense_inputs(B, Hq, Hkv, N, d, "bf16", seed=3)
    qd, kd, vd, dd = (t.to(dev) for t in (q, k, v, dout))
    o, lse = A.fwd(qd, kd, vd, True, None)
    torch.cuda.synchronize()
    out = {"status_before": A.get_device_status()}
    nbytes = lib.attn_bwd_workspace_bytes(B, Hq, N, d)
    ws = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device=dev)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    t0 = time.perf_counter()
    out["launch"] = lib.attn_bwd_main(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), dd.data_ptr(), lse.data_ptr(),
                                      dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), ws.data_ptr(), nbytes, B, Hq, Hkv,
                                      N, d, 1, 0.0, _lib.ATTN_BF16, _lib.ATTN_FLAG_DETERMINISTIC, stream)
    out["status_after_stuck_call"] = lib.attn_get_device_status(stream)
    out["seconds"] = time.perf_counter() - t0
    # the same context, a normal deterministic backward
    g = A.bwd(qd, kd, vd, o, lse, dd, True, None, out_f32=True, deterministic=True)
    torch.cuda.synchronize()
    out["status_after_normal_call"] = A.get_device_status()
    f64 = lambda t: t.detach().to("cpu", torch.float64).numpy()
    refs = oracle.bwd(f64(q), f64(k), f64(v), f64(dout), True)
    out["max_err"] = [float(np.abs(f64(a) - r).max()) for a, r in zip(g, refs)]
    print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
