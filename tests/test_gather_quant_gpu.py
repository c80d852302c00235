"""GPU checks of the row gather and the pack / quantise helpers (bit-exact)."""

import numpy as np
import pytest
import torch

import oracle
from bit_weight_only_gemv_gb300 import lib, synth
from _helpers import POISON, dev_bf16, dev_words, host_bits, host_words, poison_bf16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("v,k,t", [(50, 32, 3), (1000, 2048, 64), (777, 8960, 5),
                                   (300, 5376, 17), (10, 96, 1)])
def test_gather_bit_exact(cuda_lib, v, k, t):
    rng = np.random.default_rng(v + k + t)
    qw_h = synth.np_words(rng, (v, k // 8))
    st_h = synth.np_steps(rng, (v, k // 32), scale=rng.uniform(0.001, 10))
    ids_h = rng.integers(0, v, size=t).astype(np.int32)
    out = poison_bf16((t, k))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.embed_gather(dev_words(qw_h), dev_bf16(st_h), torch.from_numpy(ids_h).cuda(), out=out,
                     status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(host_bits(out), oracle.gather_ref(qw_h, st_h, ids_h))


def test_gather_is_the_tied_gemv_column(cuda_lib):
    rng = np.random.default_rng(1)
    v, k = 4096, 2048
    qw_h = synth.np_words(rng, (v, k // 8))
    st_h = synth.np_steps(rng, (v, k // 32))
    qw, st = dev_words(qw_h), dev_bf16(st_h)
    ids = torch.arange(v, dtype=torch.int32, device="cuda")
    table = host_bits(lib.embed_gather(qw, st, ids))
    for kk in (0, 777, k - 1):
        x_h = np.zeros((1, k), np.uint16)
        x_h[0, kk] = 0x3F80
        y = lib.gemv(qw, st, dev_bf16(x_h))
        torch.cuda.synchronize()
        assert np.array_equal(host_bits(y)[0], table[:, kk])


def test_gather_bad_id_leaves_row_unwritten(cuda_lib):
    rng = np.random.default_rng(2)
    v, k = 64, 2048
    qw_h = synth.np_words(rng, (v, k // 8))
    st_h = synth.np_steps(rng, (v, k // 32))
    ids_h = np.array([3, 64, -5, 0], np.int32)
    out = poison_bf16((4, k))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.embed_gather(dev_words(qw_h), dev_bf16(st_h), torch.from_numpy(ids_h).cuda(), out=out,
                     status=status)
    torch.cuda.synchronize()
    assert lib.STATUS[int(status.item())] == "W4_ERR_INDEX"
    b = host_bits(out)
    assert np.all(b[1] == POISON) and np.all(b[2] == POISON)
    assert np.array_equal(b[[0, 3]], oracle.gather_ref(qw_h, st_h, ids_h[[0, 3]]))


def test_pack_bit_exact_and_rejects_bad_codes(cuda_lib):
    rng = np.random.default_rng(3)
    codes = synth.np_codes(rng, (37, 96))
    qw = lib.pack(torch.from_numpy(codes).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(host_words(qw), oracle.pack_codes(codes))
    bad = codes.copy()
    bad[5, 17] = 16
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    qw2 = torch.full((37, 12), 0x5A5A5A5A, dtype=torch.int32, device="cuda")
    lib.pack(torch.from_numpy(bad).cuda(), qw=qw2, status=status)
    torch.cuda.synchronize()
    assert lib.STATUS[int(status.item())] == "W4_ERR_VALUE"
    got = host_words(qw2)
    assert got[5, 2] == 0x5A5A5A5A                 # the word holding the bad code
    want = oracle.pack_codes(codes)
    mask = np.ones_like(got, bool)
    mask[5, 2] = False
    assert np.array_equal(got[mask], want[mask])


@pytest.mark.parametrize("n,k", [(5, 32), (64, 2048), (33, 5376)])
def test_quantize_bit_exact(cuda_lib, n, k):
    rng = np.random.default_rng(n + k)
    w = (rng.standard_normal((n, k)) * 10.0 ** rng.integers(-4, 4, (n, 1))).astype(np.float32)
    w[0, :32] = 0.0
    w[1 % n, 32 % k:64 % k or 32] = 0.25
    w[-1, 3] = -w[-1, 3:35].__abs__().max() - 1.0    # a unique extreme
    w[-1, 7] = -w[-1, 3]                              # tie in magnitude, later in K
    qw, st = lib.quantize(torch.from_numpy(w).cuda())
    torch.cuda.synchronize()
    qw_ref, st_ref = oracle.quantize_ref(w)
    assert np.array_equal(host_bits(st), st_ref)
    assert np.array_equal(host_words(qw), qw_ref)
