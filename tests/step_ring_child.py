"""Child process of the weight-ring tests: runs a decode step under the launch
settings in the DG_TUNE environment variable and checks every output bitwise
against the per-op entry points.  Workload "small" (the default): rows of at
most 4 KB, so 4 KB ring stages hold a few rows each and the ring wraps
hundreds of times; "splits": phases whose rows are shared by 1, 2 and 4 warps
back to back (their slot barriers live at the same time).  Exits 0 on
success; prints the first mismatch otherwise."""
import os
import sys

import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import quantized_skinny_gemm_gb300 as dg  # noqa: E402
from quantized_skinny_gemm_gb300 import synth  # noqa: E402

DEV = torch.device("cuda:0")


SHAPES = {
    # (N, K): ragged row counts, K from one chunk to 2048 (row bytes <= 4 KB)
    "small": [(151, 8), (4097, 520), (2048, 1024), (999, 2048), (33, 1536)],
    # K = 4096: 2 warps per row; 12288 and 8960: 4; 3072: 1 (streamed)
    "splits": [(777, 4096), (300, 12288), (1000, 4096), (1536, 8960), (500, 3072),
               (999, 2048), (64, 4096)],
}


def main(workload):
    g = synth.generator(21)
    shapes = SHAPES[workload]
    keep, ops, checks = [], [], []
    for N, K in shapes:
        W = synth.normal((N, K), 0.02, g).to(DEV)
        x = synth.normal((1, K), 1.0, g).to(DEV)
        y = torch.empty(1, N, dtype=torch.float16, device=DEV)
        keep += [W, x, y]
        ops.append(dg.linear(dg.LINEAR_F16, W, 1, N, K, x=x, y=y))
        checks.append((W, x, y))
    # a RAW chain through the outputs (grid barriers) and an lm_head after it
    W1 = synth.normal((1024, 2048), 0.02, g).to(DEV)
    y1 = torch.empty(1, 1024, dtype=torch.float16, device=DEV)
    x0 = next(x for _, x, _ in checks if x.shape[1] == 2048)  # a 2048-wide input, read again
    Wh = synth.normal((7000, 1024), 0.02, g).to(DEV)
    logits = torch.empty(7000, dtype=torch.float32, device=DEV)
    token = torch.empty(1, dtype=torch.int32, device=DEV)
    keep += [W1, y1, Wh, logits, token]
    ops.append(dg.linear(dg.LINEAR_F16, W1, 1, 1024, 2048, x=x0, y=y1))
    ops.append(dg.linear(dg.LINEAR_F16, Wh, 1, 7000, 1024, x=y1, logits=logits, token=token))
    plan = dg.StepPlan(ops, keep)
    ws = torch.empty(plan.workspace_bytes(), dtype=torch.uint8, device=DEV)
    for rep in range(3):  # repeated launches reuse the workspace
        dg.decode_step_weights(plan, ws)
    torch.cuda.synchronize()
    dg.check_device_status()

    for i, (W, x, y) in enumerate(checks):
        ref = torch.empty_like(y)
        dg.gemv_f16(W, x, ref)
        torch.cuda.synchronize()
        if not torch.equal(y, ref):
            print("mismatch in op %d (%s)" % (i, tuple(W.shape)))
            return 1
    r1 = torch.empty_like(y1)
    dg.gemv_f16(W1, x0, r1)
    rl = torch.empty_like(logits)
    rt = torch.empty_like(token)
    head = dg.linear(dg.LINEAR_F16, Wh, 1, 7000, 1024, x=r1, logits=rl, token=rt)
    hws = torch.empty(dg.workspace_bytes([head]), dtype=torch.uint8, device=DEV)
    dg.lm_head_argmax(head, hws)
    torch.cuda.synchronize()
    if not torch.equal(y1, r1):
        print("mismatch in the chained op")
        return 1
    if not torch.equal(logits, rl) or int(token.item()) != int(rt.item()):
        print("mismatch in the lm_head")
        return 1
    print("OK")
    return 0


if __name__ == "__main__":
    sys.exit(main(sys.argv[1] if len(sys.argv) > 1 else "small"))
