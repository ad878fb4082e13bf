"""Decode plan bytes (layout of csrc/plan_format.h) for the host tests."""
import numpy as np

HEADER = ["magic", "version", "batch", "num_heads", "kv_dtype", "total_q", "n_units", "n_merge", "rows_cap",
          "n_part_rows", "max_pages", "req_off", "units_off", "merge_off", "total_bytes", "debug_skip_copy",
          "cta_pair", "reserved0", "reserved1", "reserved2"]
UNIT = ["b", "qrow0", "nrows", "kv_begin", "kv_end", "part_row0", "split", "n_splits", "ctx", "q", "tok0",
        "flags"]
REQ = ["ctx", "q", "tok0", "fold"]
MERGE = ["qrow0", "nrows", "part_row0", "n_splits"]


def read_plan(buf: np.ndarray) -> dict:
    w = np.frombuffer(buf.tobytes(), dtype=np.int32)
    h = dict(zip(HEADER, w[:len(HEADER)].tolist()))
    def rows(off, n, fields):
        a = w[off // 4: off // 4 + n * len(fields)].reshape(n, len(fields))
        return [dict(zip(fields, r.tolist())) for r in a]
    return {"header": h,
            "requests": rows(h["req_off"], h["batch"], REQ),
            "units": rows(h["units_off"], h["n_units"], UNIT),
            "merges": rows(h["merge_off"], h["n_merge"], MERGE)}
