"""The benchmarked decode step at full size, against the oracle.

The Llama-3.1-8B-shaped 2-bit workload (batch 1, 32 query heads over 8 KV
heads, 196,608 cached tokens), set up and launched exactly as the benchmark
sets it up and launches it: codebooks and s from the default calibration,
the whole cache encoded on the GPU by vqkv_encode from the seeded synthetic
K/V, then one vqkv_decode_append call (the new K and V rows of the step are
encoded into position 196,607 and attended in the same kernel) with the
automatic split plan, including the planner's shorter split for the CTA that
encodes the new rows.  Checked:
  * every code of the GPU-encoded cache (2 x 8 x 196,608 x 32) against the
    oracle's own encoding of the same rows: bit-exact except near-ties, which
    are counted, recorded and bounded;
  * the step's appended codes against the oracle's encoding of the new rows,
    and every other cache byte untouched;
  * O of sampled query heads against the oracle's attention over the
    oracle-encoded cache (with the oracle-encoded new rows), within 2e-3;
  * every O row inside the value codebook's range (a convex combination)."""
import numpy as np
import pytest

from oracle import vqkv_oracle as vo
from tests import helpers as H
from tests import tie_log
from vector_quantized_bit_gb300 import _build, _lib, synth

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

CHUNK = 2048   # rows per oracle job


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _gen_head(args):
    w, h = args
    return synth.keys(w, 0, h, 0, w.seq_len), synth.values(w, 0, h, 0, w.seq_len)


def _oracle_chunk(args):
    """Oracle codes of rows [r0, r1) of one (KV head, role), regenerated from
    the seed, compared with the GPU's codes of the same rows."""
    w, h, role, r0, r1, s_h, cb_h, gpu = args
    x = (synth.keys if role == 0 else synth.values)(w, 0, h, r0, r1 - r0)
    ref, d32 = vo.encode_rows(x, role, s_h if role == 0 else None, cb_h)
    ties, fails = H.check_codes(gpu, ref, d32)
    return ref.astype(np.uint8), ties, fails


def test_full_size_fused_step_against_oracle():
    import torch
    w = synth.WORKLOADS[1]
    L, Hkv, cap, mode = w.seq_len, w.Hkv, w.cap_len, w.mode
    s, kcb, vcb = H.calibrate(w)
    with H.pool(min(Hkv, 16)) as ex:
        kv = list(ex.map(_gen_head, [(w, h) for h in range(Hkv)]))
    sb = _lib.vqkv_code_bytes(mode, cap)
    codes = []
    dev_ties = []
    for role in (0, 1):
        buf = torch.zeros((1, Hkv, sb), dtype=torch.uint8, device="cuda")
        cnt = torch.zeros(1, dtype=torch.int64, device="cuda")
        x = H.dev(np.stack([kv[h][role] for h in range(Hkv)])[None])
        _lib.vqkv_encode(mode, role, x, H.dev(np.zeros(1, np.int32)), H.dev(s) if role == 0 else None,
                         H.dev(kcb if role == 0 else vcb), buf, cap, near_tie_count=cnt)
        del x
        codes.append(buf)
        dev_ties.append(cnt)
    del kv
    torch.cuda.synchronize()
    before = [c.cpu().numpy() for c in codes]

    # the step, as the benchmark runs it
    lens = synth.seq_lens(w)
    q = synth.queries(w)
    new_k = np.stack([synth.appended_keys(w, 0, h, 1) for h in range(Hkv)])[None, :, 0]
    new_v = np.stack([synth.values(w, 0, h, L - 1, 1) for h in range(Hkv)])[None, :, 0]
    out = torch.full((1, w.Hq, 128), float("nan"), dtype=torch.float16, device="cuda")
    ws = _lib.decode_workspace(mode, w.B, w.Hq, Hkv, cap, int(lens.max()))
    app_ties = torch.zeros(1, dtype=torch.int64, device="cuda")
    _lib.vqkv_decode_append(mode, H.dev(q), codes[0], codes[1], H.dev(lens.astype(np.int32)), H.dev(kcb),
                            H.dev(vcb), H.dev(s), out, ws, cap, int(lens.max()), H.dev(new_k), H.dev(new_v),
                            near_tie_count=app_ties)
    torch.cuda.synchronize()
    o = out.cpu().numpy()
    after = [c.cpu().numpy() for c in codes]
    assert np.isfinite(o).all()
    assert int(ws[:4].view(torch.int32).item()) == 0   # no device error bit

    # 1. the GPU-encoded cache against the oracle, every code
    gpu_codes = {(role, h): vo.unpack_stream_fast(before[role][0, h], mode, role, L).astype(np.uint8)
                 for role in (0, 1) for h in range(Hkv)}
    jobs = [(w, h, role, r0, min(r0 + CHUNK, L), s[h], (kcb if role == 0 else vcb)[h],
             gpu_codes[role, h][r0:r0 + CHUNK])
            for role in (0, 1) for h in range(Hkv) for r0 in range(0, L, CHUNK)]
    ref_codes = [np.empty((Hkv, L, 32), dtype=np.uint8) for _ in range(2)]
    ties = [0, 0]
    fails = [0, 0]
    with H.pool() as ex:
        for (_, h, role, r0, r1, *_), (ref, t, f) in zip(jobs, ex.map(_oracle_chunk, jobs, chunksize=4)):
            ref_codes[role][h, r0:r1] = ref
            ties[role] += t
            fails[role] += f
    n_role = Hkv * L * 32
    for role in (0, 1):
        name = f"full-size Llama-shaped cache encode, role {role}"
        tie_log.record(name, n_role, ties[role], fails[role], int(dev_ties[role].item()))
        assert fails[role] == 0, (role, ties[role], fails[role])
        assert ties[role] <= tie_log.bound(n_role)
        assert int(dev_ties[role].item()) <= tie_log.bound(n_role)

    # 2. the appended rows: codes against the oracle, nothing else written
    got_all, ref_all, d_all = [], [], []
    for role, x, cb in ((0, new_k, kcb), (1, new_v, vcb)):
        off = vo.offset_table(mode, role, L)[L - 1]
        for h in range(Hkv):
            ref, d32 = vo.encode_rows(x[0, h][None], role, s[h] if role == 0 else None, cb[h])
            got = vo.unpack_stream_fast(after[role][0, h], mode, role, L)[L - 1:L]
            got_all.append(got.reshape(-1))
            ref_all.append(ref.reshape(-1))
            d_all.append(d32.reshape(ref.size, -1))
            ref_codes[role][h, L - 1] = ref[0]
            mask = np.ones(sb, dtype=bool)
            mask[off] = False
            assert np.array_equal(after[role][0, h][mask], before[role][0, h][mask]), (role, h)
    H.check_and_record_codes("full-size fused step, appended rows", np.concatenate(got_all),
                             np.concatenate(ref_all), np.concatenate(d_all), int(app_ties.item()))

    # 3. every O row is a convex combination of value rows
    lo = vcb.astype(np.float32).min(axis=(1, 2))
    hi = vcb.astype(np.float32).max(axis=(1, 2))
    for h in range(w.Hq):
        kvh = h // w.g
        assert (o[0, h] >= lo[kvh] - 1e-2).all() and (o[0, h] <= hi[kvh] + 1e-2).all(), h

    # 4. sampled heads against the oracle's attention over its own codes
    r = np.random.default_rng(11)
    heads = sorted({(0, int(r.integers(w.Hq))) for _ in range(3)} | {(0, w.Hq - 1)})
    kc = [[ref_codes[0][h] for h in range(Hkv)]]
    vc = [[ref_codes[1][h] for h in range(Hkv)]]
    ref_o = vo.decode_attention(q, kc, vc, kcb, vcb, s, lens, heads=heads)
    for b, h in heads:
        e = vo.o_error(o[b, h], ref_o[b, h])
        assert e <= H.O_TOL, (b, h, e)
