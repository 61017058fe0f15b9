"""Worker for the stacked-layer test: the oracle's weight path applied to one
expert of one synthetic layer, in a separate (spawned) process."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def quantize_expert(seed: int, e: int, E: int, H: int, I: int):
    os.environ["ORACLE_THREADS"] = "1"
    import numpy as np

    import oracle
    from synth import inputs as S

    layer = S.Layer("stack", E, H, I, 0, 1, seed, np.zeros((0, H), np.uint16), np.zeros((0, 1), np.int32),
                    np.zeros((0, 1), np.float32))
    w13 = oracle.quantize_weight(layer.weight_bf16(e, "w13"))
    w2 = oracle.quantize_weight(layer.weight_bf16(e, "w2"))
    return e, w13, w2
