"""A short decode run on a reduced copy of a synthetic workload, for profiler captures.

The model keeps the workload's layer shapes, batch and context but only
`--layers` decoder layers (and optionally a smaller vocabulary), so that one
kernel of a given shape can be captured by a profiler with a few GB on the
device.  Steps run eagerly by default (one launch per kernel, in the order of
dec_debug_step_prefix: embed, then qkv, attention, o_proj, gate_up, down per
layer, then lm_head); `--graph` replays the captured step graph instead.

    python -m token_decode_step_gb300.profile_case --config qwen3-8b-b1 --layers 2
"""

from __future__ import annotations

import argparse
import pathlib
import sys

import torch

sys.path.insert(0, str(pathlib.Path(__file__).resolve().parent.parent))

import synthetic  # noqa: E402
from token_decode_step_gb300.torch_glue import Decoder  # noqa: E402


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--config", default="qwen3-8b-b1", choices=sorted(synthetic.WORKLOADS))
    ap.add_argument("--layers", type=int, default=2)
    ap.add_argument("--vocab", type=int, default=0, help="0 keeps the workload's vocabulary")
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--graph", action="store_true")
    ap.add_argument("--proj", type=int, default=0, choices=[0, 1, 2],
                    help="dec_config.proj_kernels: 0 auto, 1 mma.sync, 2 tcgen05 (2..32-row projections)")
    ap.add_argument("--sample", type=int, default=0,
                    help="after the steps, this many dec_sample calls on the last step's logits "
                         "(temperature 0.8, top_k 50, top_p 0.9)")
    ap.add_argument("--tps", type=int, default=1,
                    help="tokens per sequence and step (> 1: a verify step or a prefill chunk from position 0)")
    a = ap.parse_args(argv)

    kw = {"n_layers": a.layers, "steps": a.steps * a.tps}
    if a.vocab:
        kw["vocab"] = a.vocab
    wl = synthetic.WORKLOADS[a.config].replace(**kw)
    model = synthetic.generate(wl, device="cuda")
    d = Decoder(wl, model, tokens_per_seq=a.tps, proj_kernels=a.proj)
    d.set_graph_mode(a.graph)
    B = wl.batch
    rows = B * a.tps
    logits = torch.empty((rows, wl.vocab), device="cuda")
    amax = torch.empty((rows,), dtype=torch.int32, device="cuda")
    tok, pos = model["tokens"].clone(), model["positions"].clone()
    kv = synthetic.kv_buffer(model["kv"])
    if a.tps > 1:  # the same chunk of tokens from position 0 every step
        tok = torch.randint(0, wl.vocab, (rows,), dtype=torch.int32, device="cuda")
        pos = torch.zeros_like(pos)
    for i in range(a.steps):
        # the algorithmic bytes of this step's attention launches (at its mean cached length)
        mean_p = float(pos.float().mean())
        print(f"step {i}: attention algorithmic bytes per launch {d.kernel_bytes(2, mean_p):.0f}", flush=True)
        d.step(tok, pos, kv, logits, amax)
        if a.tps == 1:
            d.advance(amax, tok, pos)
    if a.sample:
        from token_decode_step_gb300 import dec as D
        prm = D.SamplingParams(temperature=0.8, top_k=50, top_p=0.9, seed=1, offset=0, offset_device=None)
        stok = torch.empty((rows,), dtype=torch.int32, device="cuda")
        for i in range(a.sample):
            prm.offset = i
            D.dec_sample(logits.data_ptr(), rows, wl.vocab, prm, stok.data_ptr(),
                         torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    st = d.device_status()
    d.close()
    print(f"profile_case {a.config} layers={a.layers} vocab={wl.vocab} steps={a.steps} "
          f"graph={a.graph} status={st}")
    return 0 if st == (0, 0) else 1


if __name__ == "__main__":
    sys.exit(main())
