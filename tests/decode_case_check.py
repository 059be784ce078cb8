"""Child-process check of the decode step against the oracle, run by
test_long_context_builds_in_child with a build choice in the environment
(PKV_WIDE, read once per process): a long-context batch on the one-head
producer-warp pass.  Exit status 0 = within tolerance."""
import sys

import numpy as np
import torch

import paged_kv_cache_211_gb300 as pkv
from paged_kv_cache_211_gb300 import workloads as wl
from gpu_helpers import assert_attention_close, compact_oracle_step, dtype_code
from pkv_testutil import bits
from test_gpu_parity import _run_step


def main() -> int:
    import __graft_entry__
    __graft_entry__.build()
    dev = torch.device("cuda", 0)
    pkv.pkv_device_status(reset=True)
    w = wl.WORKLOADS["llama7b_long"].with_(num_seqs=4, num_blocks=8200)
    inp = wl.make_inputs(w, device=dev, num_layers=1)
    ids = np.arange(w.num_seqs)
    want, kn_rows, vn_rows = compact_oracle_step(inp, ids)    # before the GPU writes anything
    out, slots = _run_step(inp, dev)
    assert pkv.pkv_device_status() == 0
    assert_attention_close(bits(out)[ids], want, dtype_code(w), "long-context step")
    print("ok")
    return 0


if __name__ == "__main__":
    sys.exit(main())
