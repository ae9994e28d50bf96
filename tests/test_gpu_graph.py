"""GPU parity of a decode step captured once in a CUDA graph and replayed.

A serving loop that runs the same batch shape every step can capture its launches
once and replay them, so that the host's launch work (argument checks, tensor-map
encoding, launch calls) is paid once instead of every step. Each decode step writes
the new row of every request at its slot_mapping entry and attends over kv_len + 1
positions ("KVCache 优化技能" §3.5, the life of kv_len). Here the graph holds:

  * the K/V write of the new rows (kv_cache_write),
  * GQA decode over the full context and over a 160-token window (tcgen05 decode,
    with its merge launched as a programmatic dependent),
  * the latent-row write and absorbed MLA decode ("KVCache 优化技能" 模式三; CTA-pair
    cluster launch plus merge).

The graph reads static device buffers. Every step the host grows the block lists with
the library's manager (pkv_manager_allocate_slots, "KV Cache 管理设计文档" §3), builds
the slots, refreshes the buffers' contents (new rows, queries, slots, block table,
lengths) and replays. Each replay is checked against the oracle's write (bit for
bit) and decode of the same step.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import block_pool_ref as bp
from oracle import kv_manager_ref as km
from oracle import paged_ref as ref
from paged_kv_cache_77_gb300 import api
from tests.gpu_cases import compare

pytestmark = pytest.mark.gpu

BS, HKV, D, H = 128, 2, 128, 8
HM, DC, DR = 16, 512, 64     # MLA: query heads, latent width, rope width
WINDOW = 160
MAXB = 5
NB = 32
STEPS = 140


def _bf16(shape, gen, scale=1.0):
    return (torch.randn(shape, generator=gen, dtype=torch.float32) * scale).to(torch.bfloat16)


def test_decode_step_captured_in_a_cuda_graph_and_replayed():
    gen = torch.Generator().manual_seed(91)
    rng = np.random.default_rng(91)
    order = rng.permutation(NB).astype(np.int32)
    lib = api.KVCacheManager([0], [NB], BS, MAXB * BS, initial_orders=[order])
    orc = km.KVCacheManager([0], [NB], BS, MAXB * BS, initial_orders=[order])
    kv_len = {0: 120, 1: 250, 2: 1, 3: 383}
    reqs = sorted(kv_len)
    R = len(reqs)

    caches = {
        "k": _bf16((NB, BS, HKV, D), gen).cuda(), "v": _bf16((NB, BS, HKV, D), gen).cuda(),
        "nope": _bf16((NB, BS, 1, DC), gen).cuda(), "rope": _bf16((NB, BS, 1, DR), gen).cuda(),
    }
    bits = {n: synth.bf16_bits(t) for n, t in caches.items()}
    row_dims = {"k": (HKV, D), "v": (HKV, D), "nope": (1, DC), "rope": (1, DR)}

    def write_eager(slots, rows):
        for a, b in (("k", "v"), ("nope", "rope")):
            api.kv_cache_write(caches[a], caches[b], rows[a].cuda(), rows[b].cuda(),
                               torch.from_numpy(slots).cuda())
        for n in rows:
            bits[n] = ref.cache_write(bits[n], synth.bf16_bits(rows[n]), slots)

    # Prompts, written eagerly.
    for r in reqs:
        n = kv_len[r]
        assert lib.allocate_slots(r, 0, n) and orc.allocate_slots(r, 0, n)
        table = lib.block_table(0, [r], MAXB)
        assert np.array_equal(table, orc.block_table(0, [r], MAXB))
        slots = api.build_slot_mapping(table, [0], [n], BS)
        write_eager(slots, {k: _bf16((n,) + d, gen) for k, d in row_dims.items()})

    # Static buffers the graph reads and writes.
    st = {
        "k_new": torch.empty((R, HKV, D), dtype=torch.bfloat16, device="cuda"),
        "v_new": torch.empty((R, HKV, D), dtype=torch.bfloat16, device="cuda"),
        "nope_new": torch.empty((R, 1, DC), dtype=torch.bfloat16, device="cuda"),
        "rope_new": torch.empty((R, 1, DR), dtype=torch.bfloat16, device="cuda"),
        "q": torch.empty((R, H, D), dtype=torch.bfloat16, device="cuda"),
        "q_nope": torch.empty((R, HM, DC), dtype=torch.bfloat16, device="cuda"),
        "q_rope": torch.empty((R, HM, DR), dtype=torch.bfloat16, device="cuda"),
        "slots": torch.empty(R, dtype=torch.int32, device="cuda"),
        "table": torch.empty((R, MAXB), dtype=torch.int32, device="cuda"),
        "lens": torch.empty(R, dtype=torch.int32, device="cuda"),
    }
    outs = {n: torch.empty((R, h, d), dtype=dt, device="cuda")
            for n, h, d, dt in (("full", H, D, torch.float32), ("win", H, D, torch.bfloat16),
                                ("mla", HM, DC, torch.float32))}
    lses = {n: torch.empty((R, o.shape[1]), device="cuda") for n, o in outs.items()}
    ws = {n: torch.empty(api.decode_workspace_size(R, H, HKV, D), dtype=torch.uint8, device="cuda")
          for n in ("full", "win")}
    ws["mla"] = torch.empty(api.mla_decode_workspace_size(R, HM), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    scale, scale_m = 1.0 / np.sqrt(D), 1.0 / np.sqrt(192.0)

    def step_launches():
        api.kv_cache_write(caches["k"], caches["v"], st["k_new"], st["v_new"], st["slots"],
                           dev_status=status)
        api.kv_cache_write(caches["nope"], caches["rope"], st["nope_new"], st["rope_new"],
                           st["slots"], dev_status=status)
        for n, w in (("full", 0), ("win", WINDOW)):
            api.paged_attention_decode(st["q"], caches["k"], caches["v"], st["table"], st["lens"],
                                       scale, w, out=outs[n], lse=lses[n], workspace=ws[n],
                                       dev_status=status)
        api.mla_paged_decode(st["q_nope"], st["q_rope"], caches["nope"], caches["rope"],
                             st["table"], st["lens"], scale_m, out=outs["mla"], lse=lses["mla"],
                             workspace=ws["mla"], dev_status=status)

    graph = None
    crossed = set()
    for step in range(STEPS):
        for r in reqs:
            ok = lib.allocate_slots(r, kv_len[r], 1)
            assert ok and ok == orc.allocate_slots(r, kv_len[r], 1), f"step {step}: request {r}"
            if kv_len[r] % BS == 0:
                crossed.add(r)
        table = lib.block_table(0, reqs, MAXB)
        assert np.array_equal(table, orc.block_table(0, reqs, MAXB))
        starts = [kv_len[r] for r in reqs]
        slots = api.build_slot_mapping(table, starts, [1] * R, BS)
        assert np.array_equal(slots, bp.slot_mapping(table, starts, [1] * R, BS))
        lens = np.array([kv_len[r] + 1 for r in reqs], dtype=np.int32)
        host = {n: _bf16(tuple(t.shape), gen) for n, t in st.items() if t.dtype == torch.bfloat16}
        for n, t in host.items():
            st[n].copy_(t)
        st["slots"].copy_(torch.from_numpy(slots))
        st["table"].copy_(torch.from_numpy(table))
        st["lens"].copy_(torch.from_numpy(lens))
        for o in outs.values():
            o.fill_(float("nan"))
        if step == 0:
            # The first step runs eagerly (it also loads the library and sets the
            # kernels' attributes); then the same launches are captured.
            step_launches()
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            snapshot = {n: t.clone() for n, t in caches.items()}
            with torch.cuda.graph(graph):
                step_launches()
            # Capture launches nothing: the caches are as the eager step left them.
            for n in caches:
                assert torch.equal(caches[n], snapshot[n]), f"capture changed {n}"
        else:
            graph.replay()
        torch.cuda.synchronize()
        for n, src in (("k", "k_new"), ("v", "v_new"), ("nope", "nope_new"), ("rope", "rope_new")):
            bits[n] = ref.cache_write(bits[n], synth.bf16_bits(host[src]), slots)
            assert np.array_equal(synth.bf16_bits(caches[n]), bits[n]), f"step {step}: cache {n}"
        q64 = ref.bf16_bits_to_f64(synth.bf16_bits(host["q"]))
        rows = list(range(R))
        for n, w in (("full", 0), ("win", WINDOW)):
            o_ref, lse_ref = ref.paged_decode(q64, bits["k"], bits["v"], table, lens, BS, scale, w)
            compare(outs[n], lses[n], o_ref, lse_ref, rows, f"step {step} decode W={w}")
        qn = ref.bf16_bits_to_f64(synth.bf16_bits(host["q_nope"]))
        qr = ref.bf16_bits_to_f64(synth.bf16_bits(host["q_rope"]))
        o_ref, lse_ref = ref.mla_decode(qn, qr, bits["nope"], bits["rope"], table, lens, BS, scale_m)
        compare(outs["mla"], lses["mla"], o_ref, lse_ref, rows, f"step {step} MLA")
        assert int(status.item()) == 0
        for r in reqs:
            kv_len[r] += 1
    assert crossed == set(reqs), crossed  # every request grew into a new block under replay
