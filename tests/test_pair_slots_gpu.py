"""The b = 4 pair tables' device slots (GB300): the encoder reads a 16-level
book's pair table from a static device slot uploaded at the book's first use,
or from its kernel parameters when the slots are taken or the first use is
inside a stream capture.  Every path must give the oracle's codes (same rule
as tests/parity.py) and the same words as each other.
"""
import numpy as np
import pytest

from parity import check_rvq

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

D = 128


@pytest.fixture(scope="module")
def vq():
    from kv_cache_quantization_turboquantrvq_gb300 import api, build
    build.build()
    api.lib()
    return api


def _books(api, n, seed):
    """n distinct 16-level books near the library's (stage-1 centroids scaled)."""
    c1, b1, c2, b2 = api.vq_rvq_codebook(D, 4)
    out = []
    for k in range(n):
        f = np.float32(1.0 + 0.004 * (k + 1) + 0.0001 * seed)
        j1 = (c1 * f).astype(np.float32)
        out.append((j1, (0.5 * (j1[1:] + j1[:-1])).astype(np.float32), c2.copy(), b2.copy()))
    return out


def _x(seed):
    from kv_cache_quantization_turboquantrvq_gb300 import synth
    return synth.kv_tensor(1, 4, 2048, D, seed, 4, 20.0)


def test_more_books_than_slots(vq, oracle_mod):
    """18 new books: the first ones take device slots, the rest (slots taken)
    read their tables from the kernel parameters; all match the oracle."""
    x = _x(901)
    xd = torch.from_numpy(x).cuda()
    for book in _books(vq, 18, 1):
        p1, p2, n = vq.vq_rvq_encode_pack(xd, 4, *book)
        torch.cuda.synchronize()
        assert vq.vq_device_error() == 0
        ora = oracle_mod.rvq_encode(x.reshape(-1, D), 4, *book)
        check_rvq(p1.cpu().numpy(), p2.cpu().numpy(), n.cpu().numpy(), ora, 4)


def test_first_use_inside_a_capture(vq):
    """A book first used inside a CUDA graph capture (no upload: the kernel
    reads the parameter copy) and then eagerly (uploaded to a slot, or the
    parameters again if the slots are taken): the same words."""
    x = torch.from_numpy(_x(902)).cuda()
    book = _books(vq, 1, 7)[0]
    p1 = torch.empty((1, 4, 2048, 16), dtype=torch.int32, device="cuda")
    p2 = torch.empty_like(p1)
    nr = torch.empty((1, 4, 2048), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            vq.vq_rvq_encode_pack(x, 4, *book, packed1=p1, packed2=p2, norms=nr, stream=s)
    g.replay()
    torch.cuda.synchronize()
    q1, q2, qn = vq.vq_rvq_encode_pack(x, 4, *book)
    q1b, q2b, qnb = vq.vq_rvq_encode_pack(x, 4, *book)  # the slot, now uploaded
    torch.cuda.synchronize()
    assert vq.vq_device_error() == 0
    for a, b in ((p1, q1), (p2, q2), (nr, qn), (q1, q1b), (q2, q2b), (qn, qnb)):
        assert torch.equal(a, b)
