"""The synthetic workloads against the shape and timing facts printed on the pages
(tests/golden/pages_facts.json, each entry cited by page and section)."""
import json
import os

from speculative_decode_verify_attn_gb300 import synth

FACTS = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_facts.json")))["facts"]


def v(name):
    return FACTS[name]["value"]


def test_layer_pattern_and_window():
    w = synth.workload_256k()
    assert w.n_full + w.n_swa == v("target_layers")
    assert w.n_swa == v("window_layers_of_40")
    assert synth.WINDOW == v("window_tokens") and synth.RING == v("ring_slots")
    assert synth.CHUNK == v("chunk_tokens")
    assert w.resident_chunks * synth.CHUNK == v("pool_tokens")
    assert w.seq_lens == [v("context_tokens")] and w.depths == [v("drafts_per_step")]
    assert w.shape.num_q_heads * w.shape.head_dim == v("hidden_size")


def test_kv_heads_fit_the_20gb_statement():
    """4 KV heads x 128 over 40 layers at 256K in 16-bit KV is ~21.5 GB: 'would need ~20 GB'."""
    s = synth.LAGUNA
    total = v("target_layers") * 2 * s.num_kv_heads * s.head_dim * 2 * v("context_tokens")
    assert abs(total / 1e9 - v("full_kv_gb_at_256k")) / v("full_kv_gb_at_256k") < 0.1
    # with 8 KV heads it would be ~43 GB and with 2 ~11 GB: neither fits the statement
    assert abs(2 * total / 1e9 - 20) / 20 > 0.5 and abs(total / 2e9 - 20) / 20 > 0.4


def test_ragged_workload():
    w = synth.workload_ragged()
    lay = v("laguna_s_layers")
    assert w.n_full == lay["global"] and w.n_swa == lay["window"] and w.num_seqs == 8
    assert set(w.depths) <= set(v("ragged_depths"))
    assert all(4000 <= L <= 200000 for L in w.seq_lens)


def test_tokens_per_step_consistent_with_acceptance():
    """At a 56% per-position match rate, E[tokens/step] = 1 + sum_{k=1..16} p^k = 2.27; the
    table's 152 tok/s x (2.4 + 13.3 + 0.8) ms = 2.51 tokens/step; within 15%."""
    p = v("acceptance_long")
    expect = 1 + sum(p ** k for k in range(1, 17))
    st = v("step_ms_after")
    implied = st["tok_s"] * (st["draft"] + st["verify"] + st["heads"]) / 1000.0
    assert abs(expect - implied) / implied < 0.15
