"""GPU parity of kv4_extend_attention (chunked-prefill / extend attention
over the FP8 prefix workspace plus the FP8 chunk) against the FP64 oracle.

The gate is the attention gate of the decode tests: per output row max-abs
error <= 2e-3 and cosine >= 0.9999 against the FP64 oracle, FP32 outputs.
Why the kernel meets it on any data: K, V and (in range) q are exact in the
f16 operands, S and O accumulate in FP32, and the softmax weight p enters
the P.V product as an f16 hi + lo pair, so what is left of p's rounding is
about 2^-22 * p (a single f16 rounding, 2^-11 * max|V|, is 0.02 on the
outlier workloads, ten times the gate, when one key dominates a row: the
peaked-attention test holds exactly that case).  bf16 outputs add one bf16
rounding of the FP32 result.
"""
import numpy as np
import pytest
import torch

import bit_paged_kv_kv4_gb300 as K
from kv4_testlib import ATOL, MIN_COS, check_close
from oracle import attention as A
from workloads import extend_q, fp8_kv_codes

pytestmark = pytest.mark.gpu


def make(lp, lc, Hq, Hkv, D, seed=0, outliers=4, oscale=10.0, device="cuda"):
    rng = np.random.default_rng(seed)
    ch = [rng.choice(D, outliers, replace=False) for _ in range(Hkv)]
    TP, TC = int(sum(lp)), int(sum(lc))
    pre, s = fp8_kv_codes(seed, max(TP, 1), Hkv, D, device, ch, oscale)
    chunk, _ = fp8_kv_codes(seed + 1, max(TC, 1), Hkv, D, device, ch, oscale, scales=s)
    q = extend_q(seed, max(TC, 1), Hq, D, device)
    i32 = lambda x: torch.tensor(x, dtype=torch.int32, device=device)
    i64 = lambda x: torch.tensor(np.concatenate([[0], np.cumsum(x)]).astype(np.int64), device=device)
    return dict(q=q, ck=chunk[0].contiguous(), cv=chunk[1].contiguous(), pk=pre[0].contiguous(),
                pv=pre[1].contiguous(), s=torch.from_numpy(s).to(device), s_host=s, lp=lp, lc=lc,
                pl=i32(lp), cp=i64(lp), cl=i32(lc), cc=i64(lc), Hq=Hq, Hkv=Hkv, D=D,
                sm=np.float32(1.0 / np.sqrt(D)))


def run(x, out_dtype=torch.float32, max_chunk_len=None, split=True):
    """With split, a workspace lets the items past the last full wave of CTAs
    be cut into key-range pieces merged by the second kernel."""
    TC = max(int(sum(x["lc"])), 1)
    out = torch.zeros((TC, x["Hq"], x["D"]), dtype=out_dtype, device="cuda")
    mc = max(x["lc"]) if max_chunk_len is None else max_chunk_len
    ws = K.alloc_extend_workspace(len(x["lc"]), mc, x["Hq"], x["D"]) if split else None
    K.kv4_extend_attention(x["q"], x["ck"], x["cv"], x["pk"], x["pv"], x["s"], x["pl"], x["cp"],
                           x["cl"], x["cc"], mc, x["sm"], out, workspace=ws)
    torch.cuda.synchronize()
    return out


def oracle(x, rows=None):
    u16 = lambda t: t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    u8 = lambda t: t.cpu().numpy()
    return A.extend_attention(u16(x["q"]), u8(x["ck"]), u8(x["cv"]), u8(x["pk"]), u8(x["pv"]),
                              x["s_host"], x["lp"], x["lc"], x["sm"], rows=rows)


def vmax(x):
    from oracle.formats import e4m3_decode
    m = max(np.abs(e4m3_decode(x["pv"].cpu().numpy())).max(), np.abs(e4m3_decode(x["cv"].cpu().numpy())).max())
    return float(m) * float(x["s_host"][1])


def check(got, want, x, what):
    return check_close(np.asarray(got, np.float64), want, atol=ATOL, min_cos=MIN_COS, what=what)


@pytest.mark.parametrize("D,Hq,Hkv,lp,lc", [
    (64, 6, 2, [0, 37, 200, 64, 5], [1, 130, 300, 128, 0]),
    (128, 4, 4, [100, 0], [257, 3]),
    (256, 24, 4, [300, 0, 1000], [200, 129, 64]),
])
@pytest.mark.parametrize("split", [False, True])
def test_ragged_batch_matches_oracle(D, Hq, Hkv, lp, lc, split):
    x = make(lp, lc, Hq, Hkv, D, seed=D)
    got = run(x, split=split).cpu().numpy()
    assert K.kv4_device_error() == 0
    want = oracle(x)
    TC = int(sum(lc))
    check(got[:TC], want[:TC], x, f"D{D}")


def test_bf16_output_and_determinism():
    x = make([70, 9], [190, 33], 8, 2, 256, seed=3)
    a = run(x, torch.bfloat16)
    b = run(x, torch.bfloat16)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    f = run(x).cpu().numpy().astype(np.float64)
    got = a.float().cpu().numpy().astype(np.float64)
    # bf16 output = the FP32 result rounded once
    ulp = np.maximum(np.abs(f), 1e-30) * 2.0 ** -8
    assert np.all(np.abs(got - f) <= ulp)
    want = oracle(x)
    check(f, want, x, "fp32 beside bf16")


@pytest.mark.parametrize("lp", [[0, 1000], [100, 70], [3000, 5]])
def test_split_pieces_match_oracle_and_whole(lp):
    # few items (B 2 x 3 query tiles x 4 heads = 24 < the SM count), so every
    # item is cut into key-range pieces: prefixes shorter than the pieces
    # (empty pieces), none, and long; rows past a chunk's end; both outputs
    x = make(lp, [257, 190], 4, 2, 128, seed=21)
    assert K.kv4_extend_workspace_bytes(2, 257, 4, 128) > 0
    got = run(x).cpu().numpy()
    assert K.kv4_device_error() == 0
    whole = run(x, split=False).cpu().numpy()
    want = oracle(x)
    TC = 257 + 190
    check(got[:TC], want[:TC], x, "pieces")
    assert np.abs(got[:TC] - whole[:TC]).max() <= 1e-5 * max(1.0, np.abs(whole).max())
    b = run(x, torch.bfloat16).float().cpu().numpy()
    assert np.all(np.abs(b[:TC] - got[:TC]) <= np.maximum(np.abs(got[:TC]), 1e-30) * 2.0 ** -8)


def test_large_prefix_many_tiles_and_rescales():
    # a long prefix whose keys grow along the sequence: the running maximum
    # keeps rising, so the lazily rescaled O path runs many times
    x = make([5000], [300], 6, 1, 128, seed=11, outliers=2, oscale=30.0)
    ramp = torch.linspace(0.1, 1.0, 5000, device="cuda").view(-1, 1, 1)
    pk = x["pk"].view(torch.float8_e4m3fn).float() * ramp
    x["pk"] = pk.to(torch.float8_e4m3fn).view(torch.uint8).contiguous()
    got = run(x).cpu().numpy()
    assert K.kv4_device_error() == 0
    check(got, oracle(x), x, "ramp prefix")


def test_peaked_attention_on_large_values():
    # Two prefix keys along the queries' own +-1 pattern (at the FP8 values 448
    # and 416) take nearly all the weight of every row; the first sets the
    # row's maximum (weight exactly 1), the second gets 2^(x2 - x1), about
    # 0.3-0.7 as the query scale varies over the rows and heads.  Their values
    # sit at the FP8 maximum (|V| = 448 s_V, tens) with different sign
    # patterns.  A weight rounded once to f16 (half an ulp: 2^-12 of it) would
    # move these outputs by up to ~5e-3, above the gate; hi + lo does not.
    x = make([200], [40], 4, 1, 128, seed=7)
    sv = float(x["s_host"][1])
    d = torch.arange(128, device="cuda")
    sign = torch.where(d % 3 == 0, -1.0, 1.0)
    alt = torch.where(d % 2 == 0, 1.0, -1.0)
    r = torch.arange(40, device="cuda").view(-1, 1, 1).float()
    hq = torch.arange(4, device="cuda").view(1, -1, 1).float()
    alpha = 0.02 * (1.0 + (r * 4 + hq) / 160.0)
    x["q"][:] = (sign * alpha).to(torch.bfloat16)
    x["pk"][123, 0] = (sign * 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    x["pk"][124, 0] = (sign * 416.0).to(torch.float8_e4m3fn).view(torch.uint8)
    x["pv"][123, 0] = (-sign * 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    x["pv"][124, 0] = (alt * 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    got = run(x).cpu().numpy()
    assert K.kv4_device_error() == 0
    want = oracle(x)
    assert np.abs(want).max() > 0.3 * 448.0 * sv            # the two large values dominate
    check(got, want, x, "peaked")


def test_oversized_chunk_and_bad_query_are_flagged():
    x = make([10], [300], 2, 1, 64, seed=5)
    run(x, max_chunk_len=128)                  # rows past the grid are not computed
    assert K.kv4_device_error() == 4           # KV4_EBOUNDS
    x = make([10], [20], 2, 1, 64, seed=6)
    x["q"][3, 1, 7] = 1.0e6                    # outside the f16 range
    run(x)
    assert K.kv4_device_error() == 1           # KV4_EINVAL
    assert K.kv4_device_error() == 0


@pytest.mark.slow
def test_full_size_chunk_of_160k_request_sampled():
    # the chunked-prefill shape of the 160K workload: an 8192-token chunk after
    # a 155,426-token prefix (request 0 of the 160K decode workload), Hq 24,
    # Hkv 4, head_dim 256; sampled rows against the oracle
    lp, lc = [155426], [8192]
    x = make(lp, lc, 24, 4, 256, seed=3)
    got = run(x)
    assert K.kv4_device_error() == 0
    rng = np.random.default_rng(0)
    rows = [(0, 0), (127, 23), (128, 5), (8191, 17), (4096, 12)] + \
        [(int(r), int(h)) for r, h in zip(rng.integers(0, 8192, 11), rng.integers(0, 24, 11))]
    want = oracle(x, rows=rows)
    g = got.cpu().numpy()
    check(np.stack([g[r, h] for r, h in rows]), np.stack([want[r, h] for r, h in rows]), x, "160K chunk")
