"""Write tests/golden/tiny_mixed.json: a tiny paged batch and its oracle result.

The stored expected values are computed here by the float64 oracle
(oracle/pkv_oracle.py) and nothing else; the inputs are the seeded synthetic
generator's output (workloads.py), stored as raw bf16 bits so the fixture does
not depend on the random generator of a particular torch version.

The batch mixes the two query shapes of a continuous batch (llm-d blog post
"What does production-grade LLM inference look like?", introduction: paged
attention plus continuous batching): a decode row (one new token) and a
prefill chunk of 3 tokens, with one padding token whose slot is -1.

Run:  python tests/golden/make_golden.py
"""

import base64
import json
import os
import sys

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle.pkv_oracle as O  # noqa: E402
from workloads import make_batch  # noqa: E402


def _b64(a: np.ndarray) -> str:
    return base64.b64encode(np.ascontiguousarray(a).tobytes()).decode()


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).numpy().view(np.uint16)


def main():
    b = make_batch([5, 21, 1], [1, 3, 0], 4, 1, seed=77, pool_factor=1.0, extra_blocks=2)
    slots = b.slot_mapping.copy()
    # pad the batch with a token that writes nothing
    q = torch.cat([b.q, b.q[:1]])
    k_new = torch.cat([b.k_new, b.k_new[:1] * 0 + 7])
    v_new = torch.cat([b.v_new, b.v_new[:1] * 0 + 7])
    slots = np.concatenate([slots, [-1]])
    kc, vc = _bits(b.k_cache), _bits(b.v_cache)
    k2, v2 = O.write(_bits(k_new), _bits(v_new), slots, kc, vc, b.page_size)
    qsl = np.concatenate([b.query_start_loc, [b.query_start_loc[-1]]]).astype(np.int32)
    lens = np.concatenate([b.seq_lens, [0]]).astype(np.int32)
    bt = np.concatenate([b.block_tables, np.full((1, b.block_tables.shape[1]), b.num_blocks)]).astype(np.int32)
    # the padding token (row 4) belongs to no sequence: qsl ends at 4
    out = O.attend(_bits(q), k2, v2, bt, lens, qsl, b.scale, 4, 1, b.page_size)
    fixture = {
        "source": "tests/golden/make_golden.py -> oracle/pkv_oracle.py (float64); "
                  "inputs from workloads.make_batch(seed=77)",
        "num_q_heads": 4, "num_kv_heads": 1, "head_dim": 128, "page_size": b.page_size,
        "num_blocks": int(b.num_blocks), "scale": b.scale,
        "seq_lens": lens.tolist(), "query_start_loc": qsl.tolist(),
        "block_tables": bt.tolist(), "slot_mapping": slots.tolist(),
        "q": _b64(_bits(q)), "k_new": _b64(_bits(k_new)), "v_new": _b64(_bits(v_new)),
        "k_cache": _b64(kc), "v_cache": _b64(vc),
        "k_cache_after": _b64(k2), "v_cache_after": _b64(v2),
        "out_f64": _b64(out), "T": int(q.shape[0]), "num_query_rows": int(qsl[-1]),
    }
    with open(os.path.join(HERE, "tiny_mixed.json"), "w") as f:
        json.dump(fixture, f, indent=0)


if __name__ == "__main__":
    main()
