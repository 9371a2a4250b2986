"""Host logic of the launch-configuration sweep and the committed table
(no GPU): the table parses, every entry is a valid configuration, classes are
unique, and the sweep's selection and writer behave as documented."""
import os
import re

from dense_gemm_12_gb300 import tune

TABLE = os.path.join(os.path.dirname(__file__), "..", "dense_gemm_12_gb300", "csrc",
                     "dispatch_table.inc")
ENTRY = re.compile(r"^\s*\{(-?\d+),\s*(\d+),\s*(\d+),\s*(\d+),\s*(\d+),\s*(-?\d+),\s*(\d+)\}")


def parse_table(text):
    sms = int(re.search(r"kTunedSms\s*=\s*(\d+);", text).group(1))
    rows = [tuple(int(x) for x in m.groups()) for m in map(ENTRY.match, text.splitlines()) if m]
    return sms, rows


def test_committed_table_is_well_formed():
    sms, rows = parse_table(open(TABLE).read())
    assert sms > 0
    assert rows and rows[-1][0] == -1, "the table ends with the sentinel"
    body = rows[:-1]
    keys = [r[:4] for r in body]
    assert len(keys) == len(set(keys)), "one entry per class"
    for is_bf16, lm, ln, lk, kernel, split, group in body:
        assert is_bf16 in (0, 1)
        assert all(0 <= v <= 31 for v in (lm, ln, lk))
        # the CTA-pair kernel is bf16's, the wide tile and stream-K are fp32's
        assert kernel in (1, 2, 3)
        assert kernel != 2 or is_bf16 == 1
        assert kernel != 3 or is_bf16 == 0
        assert 1 <= split <= 8 or (split == -1 and is_bf16 == 0)
        assert 1 <= group <= 64
        # bf16 with M <= 32 runs the decode kernel, which never reads the table
        assert not (is_bf16 and lm <= 5), "dead bf16 entry for M <= 32"


def test_sweep_grid_leaves_decode_shapes_out():
    assert min(tune.BF16_M) > 64
    assert min(tune.FP32_M) >= 128 and min(tune.FP32_NK) >= 256


def test_ceil_log2_buckets():
    assert [tune.ceil_log2(x) for x in (1, 2, 3, 4092, 4096, 4097, 8192)] == \
        [0, 1, 2, 12, 12, 13, 13]


def test_candidates_respect_kernel_and_k():
    c = list(tune.candidates(True, 64, 4096, 4096))
    assert {x["kernel"] for x in c} == {"single_cta"}          # M <= 128: no pairs
    c = list(tune.candidates(True, 1024, 4096, 128))            # 2 k-blocks
    assert {x["kernel"] for x in c} == {"single_cta", "cta_pair"}
    assert max(x["split"] for x in c) == 2
    c = list(tune.candidates(False, 4092, 4092, 4092))
    assert {x["kernel"] for x in c} == {"single_cta", "wide"}
    assert -1 in {x["split"] for x in c}                        # stream-K tail
    c = list(tune.candidates(True, 1024, 4096, 4096))
    assert {x["kernel"] for x in c if x["split"] == -1} == {"cta_pair", "single_cta"}


def test_bf16_stream_k_candidates_only_where_it_runs():
    # pair kernel on 152 SMs: 76 workers; the tail's k-blocks must reach them
    assert tune.bf16_stream_k_runs("cta_pair", 1024, 2048, 4096, 152)      # 32 items x 32
    assert not tune.bf16_stream_k_runs("cta_pair", 256, 256, 256, 152)     # 1 item x 2
    assert not tune.bf16_stream_k_runs("cta_pair", 4864, 1024, 4096, 152)  # 76 items: no tail
    assert tune.bf16_stream_k_runs("single_cta", 128, 4096, 4096, 152)     # 16 x 64
    assert not tune.bf16_stream_k_runs("single_cta", 128, 512, 256, 152)   # 2 x 4
    assert -1 not in {x["split"] for x in tune.candidates(True, 256, 256, 256)}


def _result(M, auto_ms, best_ms, is_bf16=1):
    return {"is_bf16": is_bf16, "M": M, "N": 1024, "K": 1024, "auto_ms": auto_ms,
            "best_ms": best_ms, "best": {"kernel": "cta_pair", "split": 2, "group_m": 4},
            "kernel": "cta_pair", "split": 2, "group_m": 4,
            "auto": {"kernel": "cta_pair", "split": 1, "group_m": 8}, "rejected": []}


def test_choose_needs_the_margin():
    rs = [_result(256, 1.0, 0.99), _result(512, 1.0, 0.96), _result(1024, 1.0, 1.2)]
    chosen = tune.choose(rs, 0.03)
    assert [r["M"] for r in chosen] == [512]


def test_choose_skips_the_models_own_choice():
    r = _result(512, 1.0, 0.9)
    r["auto"] = dict(r["best"])       # the model already picks the best
    assert tune.choose([r], 0.03) == []


def test_table_writer_round_trips():
    text = tune.table_lines([_result(512, 1.0, 0.9), _result(300, 2.0, 1.0, is_bf16=0)], 152,
                            "GPU", "2026-01-01")
    sms, rows = parse_table(text)
    assert sms == 152
    assert rows == [(0, 9, 10, 10, 2, 2, 4), (1, 9, 10, 10, 2, 2, 4), (-1, 0, 0, 0, 0, 0, 0)]


def test_table_writer_keeps_wide_and_stream_entries():
    r = _result(4092, 2.0, 1.5, is_bf16=0)
    r.update(kernel="wide", split=-1, group_m=8)
    sms, rows = parse_table(tune.table_lines([r], 152, "GPU", "2026-01-01"))
    assert rows[0] == (0, 12, 10, 10, 3, -1, 8)


def test_one_type_sweep_keeps_the_other_types_entries():
    # re-rendering the committed table's parsed entries of both types gives
    # the same entries back, so a sweep of one type loses none of the other's
    text = open(TABLE).read()
    kept = tune.kept_entries(text, 1) + tune.kept_entries(text, 0)
    _, rows = parse_table(text)
    _, again = parse_table(tune.table_lines(kept, 152, "GPU", "today"))
    assert sorted(again) == sorted(rows)
    assert all(e["is_bf16"] == 1 for e in tune.kept_entries(text, 1))
    rows = tune.kept_rows("| bf16 | 1x1x1 | a |\n| fp32 | 2x2x2 | b |\nother\n", 0)
    assert rows == ["| fp32 | 2x2x2 | b |"]


def test_candidates_include_every_cluster_size():
    for is_bf16 in (False, True):
        c = list(tune.candidates(is_bf16, 512, 1024, 2048))
        assert {x["split"] for x in c} >= {1, 2, 3, 4, 5, 6, 7, 8}


def test_no_bf16_entry_for_a_decode_shape(gemm_lib):
    # the class's measured shape must take the tile kernels under automatic
    # dispatch, else the entry is never read (host-only path query)
    for e in tune.kept_entries(open(TABLE).read(), 1):
        M, N, K = e["M"], e["N"], e["K"]
        assert gemm_lib.gemm_select_path(1, M, N, K, 1.0, 1 << 20, K, 1 << 20, N) != "tc_decode", \
            (M, N, K)
