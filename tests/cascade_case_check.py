"""Child-process check of cascade decode against the oracle, run by
test_cascade_suffix_splits_in_child with the split and feed choices in the
environment (PKV_WARP_ITEMS, PKV_STREAM_FEED, read once per process).  Exit
status 0 = within tolerance."""
import sys

import torch

import oracle
import paged_kv_cache_211_gb300 as pkv
from gpu_helpers import assert_attention_close
from pkv_testutil import bits
from test_cascade import _shared_case


def main() -> int:
    import __graft_entry__
    __graft_entry__.build()
    dev = torch.device("cuda", 0)
    pkv.pkv_device_status(reset=True)
    P = 12
    base = [1, 5, 16, 100, 191, 192, 193, 250, 700, 1000, 64, 300, 2, 193]
    for dtype, Hq, Hkv, D, B in (("bf16", 16, 8, 128, 128), ("f16", 32, 4, 64, 50)):
        lens = [base[i % len(base)] + (i // len(base)) * 37 for i in range(B)]
        bt, cl, tables, ln, kc, vc, q = _shared_case(dev, dtype, lens, P, Hq, Hkv, D, 23)
        code = oracle.BF16 if dtype == "bf16" else oracle.F16
        want = oracle.decode_attention(code, bits(q), bits(kc), bits(vc), tables, ln, D ** -0.5)
        out = torch.empty_like(q)
        ws = pkv.new_cascade_workspace(B, Hq, D, max(lens), P, dev)
        pkv.paged_attention_decode_cascade(q, kc, vc, bt, cl, max(lens), P, D ** -0.5, out, ws)
        torch.cuda.synchronize()
        assert pkv.pkv_device_status() == 0
        assert_attention_close(bits(out), want, code, f"cascade B={B} g={Hq // Hkv} D={D}")
    print("ok")
    return 0


if __name__ == "__main__":
    sys.exit(main())
