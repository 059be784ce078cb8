"""Child-process check of chunked prefill against the oracle, run by
test_prefill_comparison_kernel with the kernel choice in the environment (the
library reads it once per process).  Exit status 0 = within tolerance."""
import sys

import numpy as np
import torch

import oracle
import paged_kv_cache_211_gb300 as pkv
from gpu_helpers import assert_attention_close
from pkv_testutil import bits
from test_prefill import _case, _run


def main() -> int:
    import __graft_entry__
    __graft_entry__.build()
    dev = torch.device("cuda", 0)
    pkv.pkv_device_status(reset=True)
    for dtype, Hq, Hkv, D in (("bf16", 32, 8, 128), ("f16", 16, 4, 64), ("bf16", 12, 4, 128)):
        specs = [(300, 64), (33, 1), (450, 160), (17, 17), (900, 300)]
        c = _case(dev, dtype, specs, Hq, Hkv, D, seed=Hq + D + 5)
        out, want, code, _, _ = _run(c, D, dev)
        assert_attention_close(bits(out), want, code, f"comparison kernel g={Hq // Hkv} D={D}")
    print("ok")
    return 0


if __name__ == "__main__":
    sys.exit(main())
