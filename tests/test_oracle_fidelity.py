"""Fidelity of the KVarN codec against the affine comparison scheme on the
synthetic workloads (gmlx page, "Quality": kvarn keeps the output closer to
that of an fp16 cache than affine quantization at every width below 8 - by
3 to 5x at 2 to 4 bits, measured there on model outputs - and the two
converge at 8 bits). Here the output is decode attention over one KV head
with the workloads' outlier statistics, against attention on the fp16
inputs; the ratios are reported (they are smaller than the page's model-level
figures) and kvarn is required to be the closer of the two at 2 to 4 bits."""
import numpy as np
import pytest

from oracle import affine, attention, codec
from quantized_kv_cache_kvarn_gb300 import workloads as W


def _kvarn(x, bits, N=128):
    out = []
    for t in range(x.shape[0] // N):
        e = codec.encode_tile(x[t * N:(t + 1) * N], bits, 2)
        out.append(codec.dequantize(e["codes"], e["a"], e["b"], e["c"]))
    return np.concatenate(out)


def _affine(x, bits):
    return affine.dequantize(*affine.quantize(x, bits))


def _err(k, v, q, kq, vq):
    sm = 1 / np.sqrt(k.shape[1])
    ref = np.stack([attention.softmax_attention(qq, k, v, sm)[0] for qq in q])
    out = np.stack([attention.softmax_attention(qq, kq, vq, sm)[0] for qq in q])
    return np.linalg.norm(out - ref) / np.linalg.norm(ref)


def test_affine_quantiser_by_hand():
    """One group of 64: values 0..63 at 2 bits -> scale 21, offset 0, codes
    rint(x / 21); the two halves of a row quantise independently."""
    x = np.concatenate([np.arange(64.0), 1000 + 2 * np.arange(64.0)])[None, :]
    codes, scale, offset = affine.quantize(x, 2)
    np.testing.assert_array_equal(scale[0], [21.0, 42.0])
    np.testing.assert_array_equal(offset[0], [0.0, 1000.0])
    np.testing.assert_array_equal(codes[0, :64], np.clip(np.rint(np.arange(64) / 21.0), 0, 3))
    np.testing.assert_array_equal(codes[0, 64:], np.clip(np.rint(2 * np.arange(64) / 42.0), 0, 3))
    assert np.abs(affine.dequantize(codes, scale, offset) - x).max() <= 21.0


@pytest.mark.parametrize("wname", ["toy", "dense32b", "hybrid"])
def test_kvarn_is_closer_to_fp16_than_affine_at_low_widths(wname):
    heads = 6 if wname == "hybrid" else 8
    wl = W.WORKLOADS[wname].with_(num_seqs=1, num_q_heads=heads, num_kv_heads=1, context=1024)
    case = W.make_dense(wl, device="cpu")
    k, v = case.k[0, 0].double().numpy(), case.v[0, 0].double().numpy()
    q = case.q[0].double().numpy()
    rows = {}
    for b in (2, 3, 4, 6, 8):
        ea = _err(k, v, q, _affine(k, b), _affine(v, b))
        ek = _err(k, v, q, _kvarn(k, b), _kvarn(v, b))
        rows[b] = (ea, ek)
    print("\n" + wname + ": " + ", ".join(f"{b} bits affine/kvarn = {ea / ek:.2f} ({ek:.1e})"
                                          for b, (ea, ek) in rows.items()))
    for b in (2, 3, 4):
        assert rows[b][1] < rows[b][0], (b, rows[b])
    assert rows[8][0] < 0.06 and rows[8][1] < 0.06
