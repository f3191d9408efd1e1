"""Reader for the golden fixtures in tests/golden/ (written by tests/golden/make_golden.py):
'#' lines are comments (what the fixture holds and the passages that define it), one
'%params <json>' line, then '@name dim...' headers each followed by that array's values."""
import json
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
FIXTURES = ("fwd_rope_causal_d64.txt", "bwd_rope_window_alibi_d64.txt", "decode_rope_d64.txt")


def load(name):
    params, arrays, cur, shape, vals = None, {}, None, None, []

    def flush():
        if cur is not None:
            a = np.array(vals, np.float64)
            assert a.size == int(np.prod(shape)), (name, cur)
            arrays[cur] = a.reshape(shape)

    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("%params "):
                params = json.loads(line[len("%params "):])
            elif line.startswith("@"):
                flush()
                head = line[1:].split()
                cur, shape, vals = head[0], tuple(int(x) for x in head[1:]), []
            else:
                vals.extend(float(x) for x in line.split())
    flush()
    return params, arrays
