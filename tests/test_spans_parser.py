"""The per-tile timestamp reader (dit_attention_ulysses_gb300.spans) on a
synthetic recording with known spans: every figure of the summary must come
out as constructed."""
import numpy as np

from dit_attention_ulysses_gb300.spans import SPAN_WORDS, parse, summarize


def _recording():
    # 2 CTAs x 4 slots; CTA 0 records 3 pieces, CTA 1 records 2 (slot 2 empty);
    # block period 1000 cycles, PV tail 700, epilogue 2000, refill 1500
    st = np.zeros((2, 4, SPAN_WORDS), dtype=np.uint64)
    for cta, pieces in ((0, 3), (1, 2)):
        c = 10_000 * (cta + 1)
        for k in range(pieces):
            blocks = 36
            first = c
            last_p = first + 1000 * (blocks - 1)
            o_done = last_p + 700
            stored = o_done + 2000
            st[cta, k] = [5_000_000 + 17 * k + 3 * cta, first, last_p, o_done, stored, (blocks << 32) | 0]
            c = stored + 1500
    return st


def test_parse_skips_empty_slots_and_keeps_order():
    recs = parse(_recording())
    assert [(r["cta"], r["piece"]) for r in recs] == [(0, 0), (0, 1), (0, 2), (1, 0), (1, 1)]
    assert all(r["blocks"] == 36 and r["kind"] == 0 for r in recs)


def test_summary_recovers_the_constructed_spans():
    s = summarize(_recording(), sm_ghz=2.0)
    assert s["pieces"] == 5 and s["ctas"] == 2
    c = s["cycles"]
    assert c["block_period"]["p50"] == 1000 and c["pv_tail"]["p50"] == 700
    assert c["epilogue"]["p10"] == c["epilogue"]["p90"] == 2000
    assert c["refill"]["n"] == 3 and c["refill"]["p50"] == 1500       # 2 in CTA 0, 1 in CTA 1
    assert abs(s["us"]["epilogue"]["p50"] - 1.0) < 1e-12                 # 2000 cycles at 2 GHz
    assert s["first_to_last_start_us"] == (17 * 2) / 1e3                 # ns -> us


def test_block_phase_summary():
    from dit_attention_ulysses_gb300.spans import PHASE_BLOCKS, PHASE_WORDS, summarize_phases
    ph = np.zeros((3, PHASE_BLOCKS, PHASE_WORDS), dtype=np.uint64)
    steps = [0, 100, 170, 260, 900, 940, 1000]          # cumulative cycles of stamps 0..6 in a block
    for cta in range(3):
        for j in range(PHASE_BLOCKS):
            t0 = 5000 + 1500 * j
            ph[cta, j, :7] = [t0 + d for d in steps]
            ph[cta, j, 7] = t0 - 400                      # S MMAs issued 500 cycles before they are seen
            ph[cta, j, 8] = t0 + 1000 + 60                # PV issued 60 cycles after P is signalled
            ph[cta, j, 9] = t0 + 1000 + 20                # the PV issuer sees P 20 cycles after warp 0's signal
            ph[cta, j, 10] = t0 + 1000 + 30               # ... and V 10 cycles later
            ph[cta, j, 14] = t0 - 2000                    # V load issued
            ph[cta, j, 16] = t0 + 1000                    # warp 0 signals with stamp 6
            ph[cta, j, 16 + 4] = t0 + 1000 + 5            # warp 4 signals 5 cycles after warp 0
    s = summarize_phases(ph)
    assert s["blocks"] == 3 * (PHASE_BLOCKS - 1)          # every recorded block but the last (no next block)
    assert (s["wait_scores"], s["load_scores"], s["row_max"], s["exponentials"]) == (100, 70, 90, 640)
    assert (s["rescale_o"], s["store_p"], s["to_next_block"], s["period"]) == (40, 60, 500, 1500)
    assert s["s_issued_to_seen"] == 500 and s["p_signalled_to_pv_issued"] == 60
    assert (s["pv_sees_p_after_warp0"], s["pv_sees_v_after_p"], s["pv_issue_after_v"]) == (20, 10, 30)
    assert s["v_load_to_seen"] == 3030 and s["warp4_p_signalled_after_warp0"] == 5


def test_epilogue_summary():
    from dit_attention_ulysses_gb300.spans import EPI_WORDS, summarize_epilogue
    ep = np.zeros((4, EPI_WORDS), dtype=np.uint64)
    steps = [0, 300, 330, 400, 900, 930, 1000, 1500]     # cumulative cycles of stamps 0..7
    for cta in range(3):
        ep[cta] = [10000 * (cta + 1) + d for d in steps]
    s = summarize_epilogue(ep)                              # CTA 3 recorded nothing
    assert s["ctas"] == 3 and s["total"] == 1500
    assert (s["destination_row"], s["load_o_0"], s["stage_0"], s["stores_0"]) == (300, 30, 70, 500)
    assert (s["load_o_1"], s["stage_1"], s["stores_1"]) == (30, 70, 500)
