"""Replays the pages' allocator traces (tests/golden/allocator_traces.json)
against any allocator exposing alloc/incref/decref/cow/refcount/num_free/
num_shared/append.  Shared by the oracle-model and the library tests."""
import json
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_traces():
    with open(os.path.join(GOLDEN, "allocator_traces.json")) as f:
        return json.load(f)["traces"]


def replay(trace, alloc, oom_exc):
    bs = trace.get("block_size", 16)
    tables, ctx, log = {}, {}, {}
    for op in trace["ops"]:
        kind = op[0]
        if kind == "alloc":
            tables.setdefault(op[1], []).extend(alloc.alloc(op[2]))
        elif kind == "alloc_oom":
            before = alloc.num_free
            try:
                alloc.alloc(op[2])
            except oom_exc:
                pass
            else:
                raise AssertionError("expected out-of-blocks")
            assert alloc.num_free == before
        elif kind == "share":
            src = tables[op[1]][:op[3]]
            alloc.incref(src)
            tables[op[2]] = list(src) + tables.get(op[2], [])
        elif kind == "prefill":
            tables[op[1]] = []
            alloc.append(tables[op[1]], 0, op[2], bs)
            ctx[op[1]] = op[2]
        elif kind == "decode":
            for _ in range(op[2]):
                for r in op[1]:
                    alloc.append(tables[r], ctx[r], 1, bs)
                    ctx[r] += 1
        elif kind == "cow":
            old = tables[op[1]][op[2]]
            new, copied = alloc.cow(old)
            log["cow"] = (old, new, copied)
            tables[op[1]][op[2]] = new
        elif kind == "release":
            alloc.decref(tables.pop(op[1]))
        elif kind == "check_table":
            assert tables[op[1]] == op[2], (trace["name"], op, tables[op[1]])
        elif kind == "check_rc":
            for b, c in op[1].items():
                assert alloc.refcount(int(b)) == c, (trace["name"], op)
        elif kind == "check_free":
            assert alloc.num_free == op[1], (trace["name"], op, alloc.num_free)
        else:
            raise ValueError(kind)
    return tables, log


def check_expect(trace, alloc, tables, log):
    e = trace["expect"]
    for r, t in e.get("tables", {}).items():
        assert tables[r] == t, (r, tables[r], t)
    if "num_free" in e:
        assert alloc.num_free == e["num_free"]
    if "num_shared" in e:
        assert alloc.num_shared == e["num_shared"]
    if "blocks_in_use" in e:
        assert trace["num_blocks"] - alloc.num_free == e["blocks_in_use"]
    if "table_entries" in e:
        assert sum(len(t) for t in tables.values()) == e["table_entries"]
    if "cow_new_block" in e:
        assert log["cow"][1] == e["cow_new_block"] and log["cow"][2]
    if "refcounts_of_s1" in e:
        assert [alloc.refcount(b) for b in tables["s1"]] == e["refcounts_of_s1"]
