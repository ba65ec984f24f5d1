"""The seeded input generators follow the stated recipe: deterministic per seed,
unit-norm q and k rows, beta after its sigmoid, the stated spreads, the document
split of the varlen workload, balanced chunk-aligned segments."""
import torch

import kda_synth


def test_prefill_inputs_recipe_and_determinism():
    a = kda_synth.prefill_inputs(512, 3, "bf16", seed=7, z_std=1.5, A_std=0.5, init_std=0.05)
    b = kda_synth.prefill_inputs(512, 3, "bf16", seed=7, z_std=1.5, A_std=0.5, init_std=0.05)
    c = kda_synth.prefill_inputs(512, 3, "bf16", seed=8, z_std=1.5, A_std=0.5, init_std=0.05)
    for n in ("q", "k", "v", "z", "A", "beta", "init_state"):
        assert torch.equal(a[n], b[n]), n
    assert not torch.equal(a["q"], c["q"])
    assert a["q"].dtype == torch.bfloat16 and a["z"].dtype == torch.float32 and a["beta"].dtype == torch.float32
    norms = a["q"].float().norm(dim=-1)
    assert torch.allclose(norms, torch.ones_like(norms), atol=1e-2)  # unit rows, then the bf16 cast
    assert float(a["beta"].min()) > 0.0 and float(a["beta"].max()) < 1.0
    assert abs(float(a["z"].std()) - 1.5) < 0.05 and abs(float(a["v"].float().std()) - 1.0) < 0.05
    assert abs(float(a["init_state"].std()) - 0.05) < 0.005
    assert kda_synth.prefill_inputs(64, 2, "f32", seed=1)["A"].abs().max() == 0  # A_std = 0 gives A = 0


def test_varlen_documents_cover_the_tokens():
    lens = kda_synth.draw_doc_lengths(32768, 512, 8192, 3)
    assert sum(lens) == 32768 and all(1 <= n <= 8192 for n in lens) and all(n >= 512 for n in lens[:-1])
    cu = kda_synth.cu_from_lengths(lens)
    assert cu.dtype == torch.int32 and int(cu[0]) == 0 and int(cu[-1]) == 32768
    assert bool((cu[1:] >= cu[:-1]).all())
    assert kda_synth.draw_doc_lengths(32768, 512, 8192, 3) == lens  # seeded


def test_segment_bounds_are_balanced_and_chunk_aligned():
    b = kda_synth.segment_bounds(16384, 148)
    sizes = [e - s for s, e in b]
    assert b[0][0] == 0 and b[-1][1] == 16384 and all(b[i][1] == b[i + 1][0] for i in range(147))
    assert sizes.count(111) == 104 and sizes.count(110) == 44  # earlier segments one chunk longer
    assert sizes == sorted(sizes, reverse=True)


def test_decode_windows_recipe():
    w = kda_synth.decode_window(8, 5, 3, 0, 5, "f32")
    assert w["q"].shape == (8, 5, 3, 128) and w["beta"].shape == (8, 5, 3)
    n = w["k"].norm(dim=-1)
    assert torch.allclose(n, torch.ones_like(n), atol=1e-5)
    assert int(w["num_accepted"].min()) >= 0 and int(w["num_accepted"].max()) <= 4
    f = kda_synth.decode_fused_window(8, 5, 3, 0, 5, "f32")
    assert f["o_gate"].shape == (8, 5, 3, 128) and float(f["beta"].min()) < 0.0  # logits, not probabilities
    p = kda_synth.decode_fused_params(3, 5)
    assert p["conv_w"].shape == (3, 3, 128, 4) and float(p["conv_w"].abs().max()) <= 0.5
    assert kda_synth.decode_conv_state(2, 3, 5).shape == (2, 3, 3, 3, 128)
    assert torch.equal(kda_synth.decode_fused_window(8, 5, 3, 1, 5)["q"], kda_synth.decode_fused_window(8, 5, 3, 1, 5)["q"])
