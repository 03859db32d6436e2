"""One kernel family at its workload's size, a few calls, for a profiler to capture.

    python -m speculative_decoding_block_verify_gb300.profile_case CASE [--calls N] [--warmup W]

Cases (inputs generated on the device from the seeded workloads, then W untimed and N more
calls; nothing is timed or checked here - bench.py and the tests do that):

  verify_block_batch64     spec_verify_block, B = 64, k = 5, V = 129,280, bf16
                           (stats_kernel, decide_kernel, sweep_kernel, finish_kernel)
  verify_tokenwise_batch64 spec_verify_tokenwise, the same inputs
  verify_block_batch256_k9 spec_verify_block, B = 256, k = 9, V = 129,280, fp32
  verify_reduced_batch64_topk  spec_verify_block_reduced, B = 64, k = 5, V = 129,280, K = 32,768
  bias_single              dspark_markov_bias, 5 rows, rank 256, V = 129,280, bf16, with a
                           256 MB scrub before every call so that W2 is read from HBM
  walk_single              dspark_markov_walk, one stream, N = 5, rank 256, V = 129,280, bf16
  pick_adaptive128         adaptive_pick_k, B = 128, kmax = 5, H = 7168, bf16, per-stream mode
  pick_batch_adaptive128   the same in batch mode (the sort of the entries in pick_batch_kernel)
  pipeline_adaptive128     SpecPipeline.launch (pick -> verify -> counters -> step + 1)

A profiler filters the launches it captures by kernel name and skips the warm-up calls.
"""

import argparse
import sys


def _bf(torch, a, dev):
    import numpy as np
    return torch.as_tensor(np.asarray(a, np.float32), device=dev).to(torch.bfloat16)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("case")
    ap.add_argument("--calls", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=2)
    a = ap.parse_args(argv)

    import numpy as np
    import torch

    import speculative_decoding_block_verify_gb300 as sv
    from speculative_decoding_block_verify_gb300 import workloads

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    sv.lib()
    total = a.warmup + a.calls
    if a.case == "verify_reduced_batch64_topk":
        s = workloads.make_verify_inputs("batch64_topk", 3000, backend="torch", device=dev)
        out = None
        for i in range(total):
            out = sv.spec_verify_block_reduced(s["cu_drafts"], s["draft_logits"], s["t2d"], s["target_logits"],
                                               s["draft_tokens"], s["temperature"], s["kmax"], 0, i, out=out)
    elif a.case.startswith("verify_"):
        rule, name = a.case.split("_", 2)[1:]
        fn = sv.spec_verify_block if rule == "block" else sv.spec_verify_tokenwise
        s = workloads.make_verify_inputs(name, 3000, backend="torch", device=dev)
        out = None
        for i in range(total):
            out = fn(s["cu_drafts"], s["draft_logits"], s["target_logits"], s["draft_tokens"],
                     s["temperature"], s["kmax"], 0, i, out=out)
    elif a.case in ("bias_single", "walk_single"):
        inp = workloads.make_verify_inputs("single_bias", 7000)
        bias = workloads.make_bias_inputs("single_bias", 7000)
        dq = _bf(torch, inp["draft_logits"], dev)
        w1, w2 = _bf(torch, bias["W1"], dev), _bf(torch, bias["W2"], dev)
        prev = torch.as_tensor(bias["prev"], device=dev)
        if a.case == "bias_single":
            out = torch.empty(dq.shape, dtype=torch.float32, device=dev)
            scrub = torch.empty(64 << 20, dtype=torch.float32, device=dev)
            for i in range(total):
                scrub.fill_(float(i))
                sv.dspark_markov_bias(dq, prev, w1, w2, out=out)
        else:
            T = torch.as_tensor(inp["temperature"], device=dev)
            out = None
            for i in range(total):
                out = sv.dspark_markov_walk(dq.view(1, 5, -1), prev[:1].contiguous(), w1, w2, T, 0, i, out=out)
    elif a.case in ("pick_adaptive128", "pick_batch_adaptive128", "pipeline_adaptive128"):
        c = workloads.make_confidence_inputs(12)
        h, w = _bf(torch, c["hidden"], dev), _bf(torch, c["w"], dev)
        vm = torch.as_tensor(c["verify_ms"], device=dev)
        if a.case != "pipeline_adaptive128":
            pk = None
            mode = 1 if a.case == "pick_batch_adaptive128" else 0
            for _ in range(total):
                pk = sv.adaptive_pick_k(h, w, 0.0, vm, mode=mode, out=pk)
        else:
            dn = workloads.make_verify_inputs("adaptive128", 13, backend="torch", device=dev)
            B, K, V = 128, 5, dn["V"]
            pl = sv.SpecPipeline(h, w, 0.0, vm, dn["draft_logits"].view(B, K, V),
                                 dn["target_logits"].view(B, K + 1, V), dn["draft_tokens"].view(B, K),
                                 dn["temperature"], rule=1)
            for _ in range(total):
                pl.launch()
            torch.cuda.synchronize()
            pl.close()
    else:
        print(f"unknown case {a.case}", file=sys.stderr)
        return 2
    torch.cuda.synchronize()
    print(f"{a.case}: {total} calls done")
    return 0


if __name__ == "__main__":
    sys.exit(main())
