"""Run the chunked forward (or the backward) on one seeded synthetic shape a few times
(for profilers).

    python -m kimi_delta_attention_gb300.run_case --B 1 --T 4096 --H 8 --HV 8 --kernel split --calls 4
    python -m kimi_delta_attention_gb300.run_case --B 1 --T 1024 --H 8 --HV 8 --op backward --calls 3

Inputs come from ``workloads.make_inputs`` (seeded, bf16 q/k/v, fp32 g/beta; the
backward adds a seeded bf16 output gradient), and the call goes through the C ABI like
any user call.  ``--kernel`` sets KDA_CHUNK_SPLIT for the process: ``split`` = 1,
``cluster`` = 0, ``auto`` leaves the dispatch alone.
"""
import argparse
import os


def main(argv=None) -> None:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--B", type=int, default=1)
    ap.add_argument("--T", type=int, default=4096)
    ap.add_argument("--H", type=int, default=8)
    ap.add_argument("--HV", type=int, default=8)
    ap.add_argument("--K", type=int, default=128)
    ap.add_argument("--V", type=int, default=128)
    ap.add_argument("--seed", type=int, default=1)
    ap.add_argument("--calls", type=int, default=4)
    ap.add_argument("--kernel", choices=["auto", "split", "cluster"], default="auto")
    ap.add_argument("--op", choices=["forward", "backward"], default="forward")
    a = ap.parse_args(argv)
    if a.kernel != "auto":
        os.environ["KDA_CHUNK_SPLIT"] = "1" if a.kernel == "split" else "0"
    import torch

    from . import _lib, workloads
    from .builder import build
    build()
    x = workloads.make_inputs(a.B, a.T, a.H, a.HV, a.K, a.V, "bf16", seed=a.seed).to("cuda")
    if a.op == "backward":
        import numpy as np
        rng = np.random.default_rng(a.seed + 1)
        do = torch.from_numpy(rng.standard_normal(tuple(x.v.shape), dtype=np.float32)).to(torch.bfloat16).cuda()
        for _ in range(a.calls):
            grads = _lib.kda_backward(x.q, x.k, x.v, x.g, x.beta, do, x.scale)
        torch.cuda.synchronize()
        print(f"ok backward max|dq|={grads[0].abs().max().item():.4g}")
        return
    for _ in range(a.calls):
        o, _s = _lib.kda_chunk_fwd(x.q, x.k, x.v, x.g, x.beta, x.scale)
    torch.cuda.synchronize()
    name = _lib.kda_chunk_fwd_kernel_name(_lib.make_shape(x.q, x.v))
    print(f"ok kernel={name} max|o|={o.float().abs().max().item():.4g}")


if __name__ == "__main__":
    main()
