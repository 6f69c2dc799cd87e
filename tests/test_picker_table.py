"""The compiled-in picker table (measured on a GB300 by tune_picker.py)."""
import csv
import os
import re

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
PKG = os.path.join(os.path.dirname(HERE), "dense_tiled_gemm_persistent_gb300")
INC = os.path.join(PKG, "csrc", "tgemm_picker_table.inc")
CSV = os.path.join(PKG, "picker_table.csv")

ROW = re.compile(r"\{(-?\d+), (-?\d+), (-?\d+), (\d+), (\d+), \{(\d+), (\d+), (\d+), (\d+), (\d+), (\d+), "
                 r"(\d+)\}, ([0-9.]+)f\},\s*// (\w+)")


def rows():
    out = []
    for line in open(INC):
        m = ROW.match(line.strip())
        if m:
            v = [int(x) for x in m.groups()[:12]]
            out.append(dict(em=v[0], en=v[1], ek=v[2], layout=v[3], dclass=v[4], bm=v[5], bn=v[6], stages=v[7],
                            cluster_m=v[8], group_m=v[9], split_k=v[10], swap_ab=v[11], us=float(m.group(13)),
                            kind=m.group(14)))
    return out


def test_every_row_is_a_legal_configuration():
    r = rows()
    assert len(r) > 100
    seen = set()
    for e in r:
        key = (e["em"], e["en"], e["ek"], e["layout"], e["dclass"])
        assert key not in seen, key
        seen.add(key)
        assert e["dclass"] in (0, 1, 2)
        if e["dclass"] == 1:
            # FP8 operands: B stored N x K; the tile kernels or the in-cluster swap-AB kernel
            assert e["layout"] == 1 and e["swap_ab"] in (0, 2)
        if e["dclass"] == 2:
            # TF32 operands: tile kernels only, B stored N x K, more than 64 rows of A
            assert e["swap_ab"] == 0 and e["layout"] == 1 and e["em"] > 6
        if e["swap_ab"]:
            M = 1 << e["em"]
            assert M <= 128 and e["bn"] >= M and e["bm"] == 128
            if M > 64:
                assert e["swap_ab"] == 2 and e["stages"] == 6 and e["split_k"] <= 4
            if e["swap_ab"] == 2:
                # the full ring (one CTA per SM) or the half ring (two per SM)
                assert e["cluster_m"] == e["split_k"]
                assert e["stages"] in ({16: 12, 32: 10, 64: 9, 128: 6}[e["bn"]], {16: 6, 32: 5, 64: 4, 128: 3}[e["bn"]])
                if e["bn"] < 128 and e["stages"] == {16: 6, 32: 5, 64: 4}[e["bn"]]:
                    assert e["split_k"] <= {16: 8, 32: 7, 64: 4}[e["bn"]]
        else:
            assert (e["cluster_m"], e["bm"]) in ((1, 128), (2, 256), (4, 256))   # 4: two pairs sharing A
            if e["cluster_m"] == 4:
                assert e["bn"] == 256
            assert e["split_k"] == 1 or (e["split_k"] == 0 and e["cluster_m"] in (2, 4))   # 0: stream-K tail


def test_table_rows_are_the_fastest_measurement_of_their_point():
    times = {}
    for m in csv.DictReader(open(CSV)):
        key = (int(m["em"]), int(m["en"]), int(m["ek"]), int(m["layout"]), int(m.get("dclass") or 0))
        times.setdefault(key, {})[m["kind"]] = float(m["us"])
    for e in rows():
        t = times[(e["em"], e["en"], e["ek"], e["layout"], e["dclass"])]
        # the CSV rounds to 1 ns, so two kinds may tie there
        assert e["kind"] in t and t[e["kind"]] == pytest.approx(min(t.values()), abs=1e-3)
        assert e["us"] == pytest.approx(t[e["kind"]], abs=1e-3)


def test_large_square_problems_pick_the_cta_pair():
    # 256 x 256 tiles on CTA pairs: whole tiles, stream-K tail, wider raster
    # bands, or two pairs sharing A
    big = [e for e in rows() if e["em"] >= 13 and e["en"] >= 13 and e["ek"] >= 12 and e["dclass"] == 0]
    assert big and all(e["kind"] in ("pair256", "pair256sk", "pair256g16", "quad256", "quad256sk") for e in big)
    assert all(e["bm"] == 256 and e["bn"] == 256 and e["cluster_m"] in (2, 4) for e in big)
