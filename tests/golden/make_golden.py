"""Writes tests/golden/oracle_small.json: a tiny seeded input and the fp64
oracle's output for it.

The pages print no worked attention values, so this fixture is a regression
record of the oracle itself (the inputs are stored as bf16 bit patterns, so it
does not depend on any random generator).  It calls only ``oracle`` and the
seeded input generator; nothing here touches the CUDA library.

Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from dit_long_sequence_gb300 import workloads as wl  # noqa: E402

B, N, H, D, KVL, SEED = 1, 20, 1, 64, 13, 7


def main():
    q, k, v, _ = wl.make_qkv(B, N, H, D, SEED, device="cpu")
    qb, kb, vb = (wl.bf16_bits(t) for t in (q, k, v))
    O, L = oracle.attn(qb, kb, vb, key_valid_len=KVL, scale=D ** -0.5)
    doc = {
        "what": "dense bidirectional attention with a key-only mask: O = softmax(scale q k^T) v over "
                "keys j < key_valid_len, LSE = ln sum_j exp(scale q.k_j)",
        "source": "Scaling Video Generation Across NVL72 rack with TensorRT-LLM, 'Attention2D "
                  "Parallelism' / 'Local Attention'; key mask: 8 卡怎么分 token：LTX-2 序列并行的 "
                  "all2all 到底搬了什么, '构造 padding mask'",
        "written_by": "tests/golden/make_golden.py (fp64 CPU oracle only)",
        "shape": {"B": B, "N": N, "H": H, "D": D, "key_valid_len": KVL, "scale": D ** -0.5},
        "layout": "q/k/v [B,N,H,D] bf16 bits as 4-hex-digit strings, row-major; O [B,N,H,D]; LSE [B,H,N]",
        "q": " ".join(f"{x:04x}" for x in qb.ravel()),
        "k": " ".join(f"{x:04x}" for x in kb.ravel()),
        "v": " ".join(f"{x:04x}" for x in vb.ravel()),
        "O": [float(x).hex() for x in O.ravel()],
        "LSE": [float(x).hex() for x in L.ravel()],
    }
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_small.json")
    with open(out, "w") as f:
        json.dump(doc, f, indent=1)
        f.write("\n")
    print("wrote", out)


if __name__ == "__main__":
    main()
