"""The cache as the whole decode state, and writes confined to the outputs (GPU).

Checkpoint and resume: an SWA(w,s) cache holds everything a later decode
needs -- the first s tokens and the latest w-s ("No post-training, just 4
more tokens", news page, section "Research method") -- so saving it is a
tensor copy.  A decode stream resumed from a copy taken mid-stream (through
host memory, as a checkpoint file would hold it) must give the same outputs
and cache bytes, bit for bit, as the stream that never stopped.

Guards: every output of every call is placed between two guard regions filled
with a sentinel bit pattern; after the call the guards must hold the
sentinel and the output must equal that of the same call into an ordinary
tensor.  Shapes include ragged tails, short ragged sequences and split
decodes, where stores run closest to the ends of their buffers.
"""
import numpy as np
import pytest
import torch

from sliding_window_attention_prefill_gb300 import (W_INF, Cache, append_decode, build, decode,
                                                    device_error, inputs, prefill, prefill_chunk,
                                                    prefill_varlen)
from sliding_window_attention_prefill_gb300 import swa as binding

pytestmark = pytest.mark.gpu

GUARD = 8192          # elements on each side (16 KiB for 16-bit types)
SENTINEL = 0x5A3C     # an unremarkable finite bf16 / fp16 pattern


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()


@pytest.mark.parametrize("w,s,cap", [(64, 4, None), (512, 4, None), (W_INF, 0, 700)])
def test_resume_from_a_saved_cache_is_bit_identical(w, s, cap):
    B, Hq, Hkv, d, prompt, steps, cut = 4, 32, 8, 128, 300, 40, 17
    kp, vp, ks, vs, qs = inputs.decode_stream(B, Hq, Hkv, d, prompt, steps, seed=61)
    c = Cache(B, Hkv, d, w, s, max_len=cap)
    c.append(kp.cuda(), vp.cuda(), 0)
    pos = torch.empty(B, dtype=torch.int32, device="cuda")
    outs, saved = [], None
    for j in range(steps):
        if j == cut:
            saved = (c.k.cpu(), c.v.cpu())  # the checkpoint: a copy in host memory
        pos.fill_(prompt + j)
        outs.append(append_decode(qs[j].cuda(), ks[j].cuda(), vs[j].cuda(), c, pos).clone())
    c2 = Cache.from_tensors(saved[0].cuda(), saved[1].cuda(), w, s)
    for j in range(cut, steps):
        pos.fill_(prompt + j)
        o = append_decode(qs[j].cuda(), ks[j].cuda(), vs[j].cuda(), c2, pos)
        assert torch.equal(o, outs[j]), f"step {j} after resuming at {cut}"
    torch.cuda.synchronize()
    assert device_error() == 0
    assert torch.equal(c2.k, c.k) and torch.equal(c2.v, c.v)


def _guarded(shape, dtype=torch.bfloat16):
    """A tensor of `shape` inside a buffer with GUARD sentinel elements on
    each side; returns (the view, the buffer)."""
    n = int(np.prod(shape))
    buf = torch.empty(n + 2 * GUARD, dtype=dtype, device="cuda")
    buf.view(torch.int16).fill_(SENTINEL)
    return buf[GUARD:GUARD + n].view(shape), buf


def _check_guards(buf, what):
    g = buf.view(torch.int16).cpu().numpy().view(np.uint16)
    assert (g[:GUARD] == SENTINEL).all(), f"{what}: written before the output"
    assert (g[-GUARD:] == SENTINEL).all(), f"{what}: written past the output"


@pytest.mark.parametrize("B,L,Hq,Hkv,d,w,s,dt", [
    (1, 333, 32, 8, 128, 64, 4, torch.bfloat16),    # ragged tail, 112-column tiles
    (2, 200, 16, 16, 64, 512, 4, torch.float16),    # G=1, d=64
    (1, 700, 32, 8, 128, W_INF, 0, torch.bfloat16),  # 256-column tiles, shuffle epilogue
    (3, 129, 8, 1, 128, 96, 4, torch.bfloat16),     # G=8, one row past a tile
])
def test_prefill_writes_only_its_output(B, L, Hq, Hkv, d, w, s, dt):
    q, k, v = inputs.prefill_inputs(B, L, Hq, Hkv, d, seed=62, dtype=dt)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    ref = prefill(q, k, v, w, s)
    out, buf = _guarded(q.shape, dt)
    prefill(q, k, v, w, s, out=out)
    torch.cuda.synchronize()
    _check_guards(buf, "prefill")
    assert torch.equal(out, ref)


def test_varlen_writes_only_its_output():
    """Short sequences end inside a query tile: their rows go out with
    16-byte stores next to the following sequence's rows."""
    Hq, Hkv, d, w, s = 32, 8, 128, 64, 4
    lens = [1, 31, 32, 33, 200, 5]
    total = sum(lens)
    q, k, v = inputs.prefill_inputs(1, total, Hq, Hkv, d, seed=63)
    q, k, v = q[0].cuda(), k[0].cuda(), v[0].cuda()
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
    ref = prefill_varlen(q, k, v, cu, w, s)
    out, buf = _guarded(q.shape)
    prefill_varlen(q, k, v, cu, w, s, out=out)
    torch.cuda.synchronize()
    assert device_error() == 0
    _check_guards(buf, "prefill_varlen")
    assert torch.equal(out, ref)


@pytest.mark.parametrize("B,Hq,Hkv,d,w,s,prompt,cap", [
    (3, 32, 8, 128, 64, 4, 500, None),       # single-chunk items
    (2, 32, 8, 128, 512, 4, 900, None),      # several chunks, split merge
    (1, 32, 8, 128, W_INF, 0, 5000, 5200),   # many splits
    (2, 16, 16, 64, 128, 4, 100, None),      # d=64, G=1
])
def test_cache_and_decode_write_only_their_buffers(B, Hq, Hkv, d, w, s, prompt, cap):
    g = inputs.generator(64)
    kp = inputs.normal_bf16((B, prompt, Hkv, d), g).cuda()
    vp = inputs.normal_bf16((B, prompt, Hkv, d), g).cuda()
    k1 = inputs.normal_bf16((B, 1, Hkv, d), g).cuda()
    v1 = inputs.normal_bf16((B, 1, Hkv, d), g).cuda()
    q = inputs.normal_bf16((B, Hq, d), g).cuda()
    capn = cap if w == W_INF else w
    ck, kbuf = _guarded((B, Hkv, capn, d))
    cv, vbuf = _guarded((B, Hkv, capn, d))
    ck.zero_(), cv.zero_()
    c = Cache.from_tensors(ck, cv, w, s)
    ref_c = Cache(B, Hkv, d, w, s, max_len=cap)
    pos = torch.full((B,), prompt, dtype=torch.int32, device="cuda")
    nws = binding.decode_workspace_bytes(B, Hq, Hkv, d, capn, w)
    ws, wbuf = _guarded((max(nws, 16) // 2,))
    c.append(kp, vp, 0)
    ref_c.append(kp, vp, 0)
    out, obuf = _guarded((B, Hq, d))
    append_decode(q, k1, v1, c, pos, out=out, workspace=ws.view(torch.uint8) if nws else None)
    ref = append_decode(q, k1, v1, ref_c, pos)
    out2, obuf2 = _guarded((B, Hq, d))
    decode(q, c, pos, out=out2, workspace=ws.view(torch.uint8) if nws else None)
    torch.cuda.synchronize()
    assert device_error() == 0
    for b_, what in [(kbuf, "cache k"), (vbuf, "cache v"), (wbuf, "workspace"), (obuf, "append_decode o"),
                     (obuf2, "decode o")]:
        _check_guards(b_, what)
    assert torch.equal(ck, ref_c.k) and torch.equal(cv, ref_c.v)
    assert torch.equal(out, ref) and torch.equal(out2, ref)


def test_chunked_prefill_writes_only_its_buffers():
    B, Hq, Hkv, d, w, s, n = 2, 32, 8, 128, 96, 4, 150
    q, k, v = inputs.prefill_inputs(B, 3 * n, Hq, Hkv, d, seed=65)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    ck, kbuf = _guarded((B, Hkv, w, d))
    cv, vbuf = _guarded((B, Hkv, w, d))
    ck.zero_(), cv.zero_()
    c = Cache.from_tensors(ck, cv, w, s)
    ref_c = Cache(B, Hkv, d, w, s)
    nws = binding.prefill_chunk_workspace_bytes(B, n, Hkv, d, w, 2 * n)
    ws, wbuf = _guarded((nws // 2,))
    for j in range(3):
        sl = slice(j * n, (j + 1) * n)
        qs, ks_, vs_ = q[:, sl].contiguous(), k[:, sl].contiguous(), v[:, sl].contiguous()
        out, obuf = _guarded(qs.shape)
        prefill_chunk(qs, ks_, vs_, c, j * n, out=out, workspace=ws.view(torch.uint8))
        ref = prefill_chunk(qs, ks_, vs_, ref_c, j * n)
        torch.cuda.synchronize()
        _check_guards(obuf, f"chunk {j} o")
        assert torch.equal(out, ref), f"chunk {j}"
    for b_, what in [(kbuf, "cache k"), (vbuf, "cache v"), (wbuf, "workspace")]:
        _check_guards(b_, what)
    assert torch.equal(ck, ref_c.k) and torch.equal(cv, ref_c.v)
