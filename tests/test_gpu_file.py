"""Packed-weight files end to end on the GPU: matrices packed on the GPU, written to a file,
loaded back (CRC-checked) into fresh device buffers, give the oracle's packed bytes and a
matvec within the library bound; a damaged section is refused and nothing is copied."""
import numpy as np
import pytest

pytestmark = [pytest.mark.gpu, pytest.mark.filterwarnings("ignore::RuntimeWarning")]

RTOL = 2e-3


@pytest.fixture(scope="module")
def env():
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import quantized_gemv_unpack_gb300 as q
    assert torch.cuda.is_available()
    return q, torch, torch.device("cuda:0")


def test_file_load_then_matvec(env, tmp_path):
    q, torch, dev = env
    from oracle import int4, ternary
    from oracle.matvec import matvec_bf16x
    from quantized_gemv_unpack_gb300 import synth
    g = synth.rng(2024)
    mats = [("blk.0.attn_q", q.QMV_TERNARY2, ternary, q.qmv_pack_ternary, 320, 1280),
            ("blk.0.ffn_down", q.QMV_INT4, int4, q.qmv_pack_int4, 96, 3072),
            ("blk.0.ffn_up", q.QMV_TERNARY2_LUT, ternary, q.qmv_pack_ternary, 200, 1024)]
    items, ws = [], {}
    for name, fmt, ref, pack, N, K in mats:
        w = synth.student_t4(g, (N, K))
        d = q.qmv_pack_desc(fmt, N, K)
        p = torch.empty(d.total_bytes, dtype=torch.uint8, device=dev)
        pack(d, torch.from_numpy(w).to(dev), p)
        items.append((name, d, p.cpu().numpy()))
        ws[name] = w
    path = str(tmp_path / "model.qmv")
    q.qmv_file_write(path, items)
    with q.QmvFile(path) as f:
        for name, fmt, ref, _, N, K in mats:
            i = f.find(name)
            _, d = f.tensor(i)
            buf = torch.full((d.total_bytes,), 0xAB, dtype=torch.uint8, device=dev)
            f.load(i, buf)
            torch.cuda.synchronize()
            qq, _, s16 = ref.quantize(ws[name])
            packed_ref = ref.pack_lut(qq, s16) if fmt == q.QMV_TERNARY2_LUT else ref.pack(qq, s16)
            assert np.array_equal(buf.cpu().numpy(), np.frombuffer(packed_ref, np.uint8)), name
            M = 1 if fmt == q.QMV_TERNARY2_LUT else 3
            xb = synth.activations_bf16(g, (M, K))
            x = torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16)
            y = torch.full((M, N), float("nan"), device=dev)
            (q.qmv_run_int4 if fmt == q.QMV_INT4 else q.qmv_run_ternary)(d, buf, x, y)
            assert q.qmv_check_status() == 0
            yr, B = matvec_bf16x(ref.dequant(qq, s16), xb)
            assert np.all(np.abs(y.cpu().numpy() - yr) <= RTOL * B), name


def test_file_load_refuses_a_damaged_section(env, tmp_path):
    q, torch, dev = env
    g = np.random.default_rng(3)
    d = q.qmv_pack_desc(q.QMV_INT4, 64, 512)
    buf = g.integers(0, 256, size=d.total_bytes, dtype=np.uint8)
    path = str(tmp_path / "bad.qmv")
    q.qmv_file_write(path, [("w", d, buf)])
    with open(path, "rb") as fh:
        data0 = int.from_bytes(fh.read(64)[24:32], "little")
    with open(path, "r+b") as fh:
        fh.seek(data0 + 100)
        b = fh.read(1)
        fh.seek(data0 + 100)
        fh.write(bytes([b[0] ^ 1]))
    dst = torch.zeros(d.total_bytes, dtype=torch.uint8, device=dev)
    with q.QmvFile(path) as f:
        with pytest.raises(q.QmvError) as e:
            f.load(0, dst)
        assert e.value.status == q.QMV_ERR_CORRUPT
    torch.cuda.synchronize()
    assert int(dst.sum()) == 0                              # nothing was copied
