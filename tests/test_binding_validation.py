"""The Python binding refuses malformed tensors before it marshals a pointer:
the kernels trust the sizes they are given, so a wrong dtype or length must
never reach them.  CPU tensors suffice (no check here needs the library)."""
import pytest
import torch

import paged_kv_cache_211_gb300 as pkv

B, Hq, Hkv, D, NB, MB = 3, 8, 2, 64, 10, 4
bf = torch.bfloat16


def _decode_args(**over):
    a = dict(q=torch.zeros(B, Hq, D, dtype=bf), k_new=torch.zeros(B, Hkv, D, dtype=bf),
             v_new=torch.zeros(B, Hkv, D, dtype=bf), k_cache=torch.zeros(NB, 16, Hkv, D, dtype=bf),
             v_cache=torch.zeros(NB, 16, Hkv, D, dtype=bf),
             block_tables=torch.zeros(B, MB, dtype=torch.int32),
             context_lens=torch.ones(B, dtype=torch.int32), max_context_len=64,
             scale=D ** -0.5, out=torch.zeros(B, Hq, D, dtype=bf),
             workspace=torch.zeros(1024, dtype=torch.uint8))
    a.update(over)
    return a


@pytest.mark.parametrize("over,msg", [
    (dict(slot_mapping_out=torch.zeros(B, dtype=torch.int32)), "slot_mapping_out must be int64"),
    (dict(slot_mapping_out=torch.zeros(B - 1, dtype=torch.int64)), "slot_mapping_out must be int64"),
    (dict(v_cache=torch.zeros(NB, 16, Hkv, D, dtype=torch.float16)), "share one dtype"),
    (dict(block_tables=torch.zeros(B * MB, dtype=torch.int32)), "block_tables must be int32"),
    (dict(block_tables=torch.zeros(B, MB, dtype=torch.int64)), "block_tables must be int32"),
    (dict(context_lens=torch.ones(B, dtype=torch.int64)), "context_lens must be int32"),
    (dict(k_new=torch.zeros(B, Hkv, D, dtype=torch.float16)), "k_new/v_new must be shaped"),
    (dict(v_new=torch.zeros(B, Hkv + 1, D, dtype=bf)), "k_new/v_new must be shaped"),
])
def test_decode_step_refuses(over, msg):
    with pytest.raises(ValueError, match=msg):
        pkv.paged_kv_decode_step(**_decode_args(**over))


def test_cascade_step_refuses_a_short_slot_output():
    a = _decode_args(slot_mapping_out=torch.zeros(1, dtype=torch.int64))
    with pytest.raises(ValueError, match="slot_mapping_out must be int64"):
        pkv.paged_kv_decode_step_cascade(a["q"], a["k_new"], a["v_new"], a["k_cache"],
                                         a["v_cache"], a["block_tables"], a["context_lens"],
                                         a["max_context_len"], 1, a["scale"], a["out"],
                                         a["workspace"], a["slot_mapping_out"])


def test_layers_step_refuses_mixed_dtypes():
    L = 2
    with pytest.raises(ValueError, match="share one dtype"):
        pkv.paged_kv_decode_step_layers(
            torch.zeros(L, B, Hq, D, dtype=bf), torch.zeros(L, B, Hkv, D, dtype=bf),
            torch.zeros(L, B, Hkv, D, dtype=bf), torch.zeros(L, NB, 16, Hkv, D, dtype=bf),
            torch.zeros(L, NB, 16, Hkv, D, dtype=torch.float16),
            torch.zeros(B, MB, dtype=torch.int32), torch.ones(B, dtype=torch.int32), 64,
            D ** -0.5, torch.zeros(L, B, Hq, D, dtype=bf), torch.zeros(1024, dtype=torch.uint8))


def test_prefill_refuses_bad_row_offsets_and_tables():
    R = 5
    q, out = torch.zeros(R, Hq, D, dtype=bf), torch.zeros(R, Hq, D, dtype=bf)
    kc = torch.zeros(NB, 16, Hkv, D, dtype=bf)
    bt, cl = torch.zeros(B, MB, dtype=torch.int32), torch.ones(B, dtype=torch.int32)
    with pytest.raises(ValueError, match="cu_q_lens must be int32"):
        pkv.paged_attention_prefill(q, kc, kc.clone(), bt, cl,
                                    torch.zeros(B + 1, dtype=torch.int64), 2, 0.1, out)
    with pytest.raises(ValueError, match="block_tables must be int32"):
        pkv.paged_attention_prefill(q, kc, kc.clone(), bt[:2], cl,
                                    torch.zeros(B + 1, dtype=torch.int32), 2, 0.1, out)


def test_cache_writes_refuse_mismatched_rows_and_ids():
    kc = torch.zeros(NB, 16, Hkv, D, dtype=bf)
    kn = torch.zeros(4, Hkv, D, dtype=bf)
    with pytest.raises(ValueError, match="k_new/v_new must be shaped"):
        pkv.reshape_and_cache(kn, torch.zeros(3, Hkv, D, dtype=bf), kc, kc.clone(),
                              torch.zeros(4, dtype=torch.int64))
    with pytest.raises(ValueError, match="pools must have k_new's dtype"):
        pkv.reshape_and_cache(kn, kn.clone(), kc.half(), kc.half(),
                              torch.zeros(4, dtype=torch.int64))
    with pytest.raises(ValueError, match="slot_mapping must be int64"):
        pkv.paged_kv_slot_mapping(torch.zeros(B, MB, dtype=torch.int32),
                                  torch.ones(B, dtype=torch.int32), NB,
                                  slot_mapping=torch.zeros(B, dtype=torch.int32))
    with pytest.raises(ValueError, match="block id lists"):
        pkv.paged_kv_copy_blocks(kc, kc.clone(), torch.zeros(2, dtype=torch.int32),
                                 torch.zeros(2, dtype=torch.int64))


def test_host_step_refuses_a_short_new_row_buffer():
    a = _decode_args()
    with pytest.raises(ValueError, match="k_new/v_new must be shaped"):
        pkv.paged_kv_decode_step_host(a["q"], a["k_new"][:2], a["v_new"], a["block_tables"],
                                      a["context_lens"], a["out"],
                                      torch.zeros(1024, dtype=torch.uint8), a["k_cache"],
                                      a["v_cache"], 64, a["scale"], a["workspace"])
