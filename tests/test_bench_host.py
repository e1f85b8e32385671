"""Host logic of bench.py (CPU only): the identity under which an ncu traffic
summary stays attached to the decode kernel, and the reading of the committed
summaries."""
import re

import bench


def test_code_identity_ignores_comments_and_blank_lines():
    src = "int f(int x)\n{\n    return x + 1;  // one more\n}\n"
    same = "/* a header */\nint f(int x)\n{\n\n    return x + 1;\n}   \n// trailing note\n"
    other = "int f(int x)\n{\n    return x + 2;  // one more\n}\n"
    assert bench._code_only(src) == bench._code_only(same)
    assert bench._code_only(src) != bench._code_only(other)
    assert "one more" not in bench._code_only(src)


def test_committed_traffic_summaries_are_readable():
    """Each traffic summary names the decode code it was taken on (a 16-hex
    identity) and a per-launch DRAM byte count; the bench reports that count
    only while the current code has the same identity."""
    import os
    h = bench.decode_source_hash()
    assert re.fullmatch(r"[0-9a-f]{16}", h)
    for cfg in (2, 3, 5):
        txt = open(os.path.join(bench.ROOT, "profiles", f"decode_config{cfg}_traffic.md")).read()
        sha = re.search(r"kernel_source_sha:\s*([0-9a-f]{16})", txt)
        tr = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", txt)
        assert sha and tr and int(tr.group(1)) > 0
        assert (bench.profiled_traffic(cfg) is not None) == (sha.group(1) == h)
