"""GPU parity of the prefill path: full-layer double buffering from the shared slot pool
(residency compared with the oracle after every layer), routing of the chunk, the
tcgen05 grouped GEMMs and the fixed-order combine (outputs vs the float64 oracle)."""
import numpy as np
import pytest

import synth
from ftharness import Run, prefill_step

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__ as g

    g.build()


def test_prefill_small_every_token_and_decode_after():
    """4 layers, 16 experts, top-2, 200 tokens (ragged tiles), 40 slots; then decode."""
    w = synth.prefill().with_(n_layers=4, n_experts=16, top_k=2, hidden=256, inter=128, cache_slots=40,
                              prefill_tokens=200)
    with Run(w, max_prefill_tokens=256) as r:
        for l in range(w.n_layers):
            prefill_step(r, 0, l, 200)
        # decode afterwards uses what prefill left resident
        dw = w.with_(logits="normal")
        r.w = dw
        for s in range(4):
            for l in range(w.n_layers):
                r.step(s, l, check_out=True)
        r.compare_state()
        print("max rel err", r.max_err)


def test_prefill_chunk_break_restores_streamed_buffer():
    """A decode step while layer 3 streams into the buffer that still holds layer 1."""
    w = synth.prefill().with_(n_layers=6, n_experts=16, top_k=2, hidden=256, inter=128, cache_slots=48,
                              prefill_tokens=64)
    with Run(w, max_prefill_tokens=64) as r:
        for l in range(3):
            prefill_step(r, 0, l, 64)
        dw = w.with_(logits="normal")
        r.w = dw
        for l in range(w.n_layers):
            r.step(0, l, check_out=True)        # layer 1's experts must still be intact
        r.w = w
        for l in range(2, 6):                   # new chunk starting mid-model
            prefill_step(r, 1, l, 64)
        r.compare_state()


def test_prefill_35b_expert_shape_sampled_tokens():
    """H 2048, I 512, 256 experts top-8, 1024 tokens, 3 layers: sampled token rows."""
    w = synth.prefill().with_(n_layers=3, cache_slots=700, prefill_tokens=1024)
    rng = np.random.default_rng(0)
    with Run(w, max_prefill_tokens=1024) as r:
        for l in range(w.n_layers):
            prefill_step(r, 0, l, 1024, check_tokens=sorted(rng.choice(1024, 24, replace=False)))
        print("max rel err", r.max_err)


def test_prefill_35b_full_chunk_second_n_tiles():
    """The prefill workload's own chunk: 8192 tokens, 35B-A3B expert shape, uniform logits
    (n_e = 256 +- 16 pairs per expert), 2 layers.  An expert with more than 256 pairs takes
    two N tiles; its tokens are in ascending order, so its last token's pair sits in the
    second tile.  The sampled rows hold, for each such expert, its last token (up to 64 of
    them), plus the first and last token of the chunk and random ones; residency after each
    layer is compared in full."""
    import oracle as O

    T = 8192
    w = synth.prefill().with_(n_layers=2, cache_slots=700, prefill_tokens=T)
    rng = np.random.default_rng(1)
    with Run(w, max_prefill_tokens=T) as r:
        n_second = 0
        for l in range(w.n_layers):
            sel, _ = O.route(synth.prefill_logits(w, 0, l, T), w.top_k)
            n_e = np.bincount(sel.reshape(-1), minlength=w.n_experts)
            big = np.nonzero(n_e > 256)[0]
            assert len(big) > 0
            last = sorted({int(np.nonzero((sel == e).any(axis=1))[0].max()) for e in big})
            n_second += len(last)
            pick = rng.choice(last, min(64, len(last)), replace=False).tolist()
            tokens = sorted(set(pick) | {0, T - 1} | set(rng.choice(T, 16, replace=False).tolist()))
            prefill_step(r, 0, l, T, check_tokens=tokens)
        assert r.F.ft_moe_get_stats(r.h).error_word == 0
        print(f"max rel err {r.max_err:.2e}; experts with a second N tile: {n_second}")


def test_prefill_with_shared_expert():
    w = synth.decode_bf16().with_(n_layers=3, n_experts=32, cache_slots=70, logits="uniform", prefill_tokens=300)
    with Run(w, max_prefill_tokens=300) as r:
        for l in range(w.n_layers):
            prefill_step(r, 0, l, 300, check_tokens=list(range(0, 300, 7)))


@pytest.mark.parametrize("slots", [31, 6])
def test_prefill_on_demand_small_pool_then_decode(slots):
    """Pools smaller than two full layers (16 experts, top-2): 31 slots load each layer's
    misses in one wave, 6 slots in waves of at most 6.  Residency after every layer and
    every output row are compared with the oracle; decode steps follow on what is left."""
    w = synth.prefill().with_(n_layers=4, n_experts=16, top_k=2, hidden=256, inter=128, cache_slots=slots,
                              prefill_tokens=200)
    with Run(w, max_prefill_tokens=256) as r:
        for l in range(w.n_layers):
            prefill_step(r, 0, l, 200)
        for l in range(w.n_layers):  # a second chunk: some experts are now hits
            prefill_step(r, 1, l, 120)
        r.compare_state()
        r.w = w.with_(logits="normal")
        for s in range(3):
            for l in range(w.n_layers):
                r.step(s, l, check_out=True)
        r.compare_state()
        print(f"slots {slots}: max rel err {r.max_err:.2e}")


def test_prefill_on_demand_capacity_error_changes_nothing():
    """One slot: after a layer, its last expert is resident; a chunk that uses it and
    another expert has no slot for the miss, so the call fails and no state changes."""
    w = synth.prefill().with_(n_layers=2, n_experts=16, top_k=2, hidden=256, inter=128, cache_slots=1,
                              prefill_tokens=64)
    with Run(w, max_prefill_tokens=64) as r:
        import torch

        prefill_step(r, 0, 0, 64)
        r.compare_state()
        u = int(r.sim.owner[0])  # the one slot holds the layer's last loaded expert
        assert u >= 0
        e_res = u % w.n_experts
        z = torch.full((8, 16), -4.0, dtype=torch.float32, device="cuda")
        z[:, e_res] = 5.0
        z[:, (e_res + 1) % 16] = 4.0  # every token: the resident expert and one more
        x = torch.zeros((8, 256), dtype=torch.int16, device="cuda")
        o = torch.empty((8, 256), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        with pytest.raises(r.F.FtError) as e:
            r.F.ft_moe_prefill_chunk(r.h, 0, 8, x, z, o)
        assert e.value.status == r.F.FT_ERR_CAPACITY
        r.compare_state()  # unchanged: the oracle was not stepped


def test_prefill_double_buffer_off_same_results():
    """The ablation switch (second buffer off: each layer loads at its own call) changes
    timing only: residency after every layer and every output row equal the oracle, and
    the outputs equal those of the double-buffered run bit for bit."""
    w = synth.prefill().with_(n_layers=4, n_experts=16, top_k=2, hidden=256, inter=128, cache_slots=40,
                              prefill_tokens=200)
    outs = {}
    for overlap in (True, False):
        with Run(w, max_prefill_tokens=256) as r:
            r.F.ft_moe_set_prefill_overlap(r.h, overlap)
            for l in range(w.n_layers):
                outs[overlap, l] = prefill_step(r, 0, l, 200)
            r.compare_state()
    for l in range(w.n_layers):
        np.testing.assert_array_equal(outs[True, l], outs[False, l])


QUANT = [synth.W_FP8_E4M3_B128, synth.W_NVFP4, synth.W_MXFP4]


@pytest.mark.parametrize("wtype", QUANT)
def test_prefill_quantized_small_every_token_then_decode(wtype):
    """FP8 / NVFP4 / MXFP4 experts through the prefill grouped GEMM: weights are decoded and
    block-scaled into BF16 tiles in shared memory before the tensor-core product.  4 layers,
    16 experts top-2, 200 tokens (ragged tiles), H 512, I 128, 40 slots; every output row
    against the float64 oracle, residency after every layer; decode steps afterwards."""
    w = synth.prefill().with_(wtype=wtype, n_layers=4, n_experts=16, top_k=2, hidden=512, inter=128,
                              cache_slots=40, prefill_tokens=200)
    with Run(w, max_prefill_tokens=256) as r:
        for l in range(w.n_layers):
            prefill_step(r, 0, l, 200)
        r.w = w.with_(logits="normal")
        for s in range(3):
            for l in range(w.n_layers):
                r.step(s, l, check_out=True)
        r.compare_state()
        print(f"wtype {wtype}: max rel err {r.max_err:.2e}")


@pytest.mark.parametrize("wtype,T", [(synth.W_FP8_E4M3_B128, 8192), (synth.W_NVFP4, 1024)])
def test_prefill_quantized_35b_expert_shape(wtype, T):
    """The prefill chunk's expert shape (H 2048, I 512, 256 experts top-8, uniform logits)
    with FP8 (the full 8192-token chunk, so routed experts take two N tiles) and NVFP4
    experts, 2 layers; sampled rows include each two-tile expert's last token."""
    import oracle as O

    w = synth.prefill().with_(wtype=wtype, n_layers=2, cache_slots=700, prefill_tokens=T)
    rng = np.random.default_rng(2)
    with Run(w, max_prefill_tokens=T) as r:
        for l in range(w.n_layers):
            sel, _ = O.route(synth.prefill_logits(w, 0, l, T), w.top_k)
            n_e = np.bincount(sel.reshape(-1), minlength=w.n_experts)
            last = sorted({int(np.nonzero((sel == e).any(axis=1))[0].max()) for e in np.nonzero(n_e > 256)[0]})
            pick = rng.choice(last, min(32, len(last)), replace=False).tolist() if last else []
            tokens = sorted(set(pick) | {0, T - 1} | set(rng.choice(T, 16, replace=False).tolist()))
            prefill_step(r, 0, l, T, check_tokens=tokens)
        assert r.F.ft_moe_get_stats(r.h).error_word == 0
        print(f"wtype {wtype} T {T}: max rel err {r.max_err:.2e}")
