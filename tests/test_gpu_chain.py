"""Back-to-back GEMMs on one stream with data dependences between them.

Consecutive launches overlap their set-up (programmatic dependent launch);
every global-memory access of a kernel comes after it has waited for the
previous kernel of the stream.  These cases would read stale or overwritten
data if that wait were missing or misplaced:

* read after write: the second GEMM's A is the first GEMM's output;
* write after read: the second GEMM overwrites the first GEMM's input;
* a chain of four dependent products, repeated without synchronisation.

Integer-valued inputs keep every intermediate exactly representable, so the
results are compared bit for bit with the oracle."""
import pytest
import torch

import dense_gemm_blackwell_gb300 as dg
import oracle
from parity import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    dg.build()
    torch.cuda.init()


def ints(shape, seed, lo=-2, hi=2):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, shape, generator=g).to(torch.bfloat16)


def ref(A, B):
    M, K = A.shape
    N = B.shape[0]
    d, s = oracle.gemm(A, B, M=M, N=N, K=K, dtype_a="bf16", dtype_b="bf16")
    return d[0], s[0]


def plan(M, N, K, out=dg.GEMM_BF16, **kw):
    return dg.Plan(dg.make_desc(M, N, K, dtype_a=dg.GEMM_BF16, dtype_d=out, **kw))


@pytest.mark.parametrize("flags", [0, dg.GEMM_FLAG_CTA_GROUP_2 | dg.GEMM_FLAG_STAGE_K2])
def test_read_after_write(flags):
    """C = A B^T, then E = C F^T with C still being written when E's kernel is
    launched; |C| <= 2 * 2 * 64 = 256 is exact in bf16."""
    M, N, K = 2048, 1536, 64
    A, B = ints((M, K), 1), ints((N, K), 2)
    F = ints((512, N), 3, -1, 1)
    dA, dB, dF = A.cuda(), B.cuda(), F.cuda()
    dC = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    dE = torch.empty(M, 512, dtype=torch.float32, device="cuda")
    with plan(M, N, K) as p1, plan(M, 512, N, out=dg.GEMM_F32, flags=flags) as p2:
        for _ in range(3):
            dC.fill_(float("nan"))
            dE.fill_(float("nan"))
            p1.run(dA, dB, dC)
            p2.run(dC, dF, dE)
        torch.cuda.synchronize()
        assert p1.sync_status()[0] == dg.GEMM_OK and p2.sync_status()[0] == dg.GEMM_OK
    C, _ = ref(A, B)
    Cb = torch.tensor(C).to(torch.bfloat16)
    assert torch.equal(Cb.float(), torch.tensor(C).float())      # exact in bf16
    E, sE = ref(Cb, F)
    r = compare(dE.double().cpu().numpy(), E, sE, "f32", 0.0, exact=True)
    assert r["ok"], r


def test_write_after_read():
    """D1 = X B^T, then X is overwritten by a second product: D1 must see the
    old X."""
    M, N, K = 1024, 1024, 128
    X, B = ints((M, K), 11), ints((N, K), 12)
    Y, Z = ints((M, 256), 13), ints((K, 256), 14, -1, 1)
    dX, dB, dY, dZ = X.cuda(), B.cuda(), Y.cuda(), Z.cuda()
    dD1 = torch.empty(M, N, dtype=torch.float32, device="cuda")
    with plan(M, N, K, out=dg.GEMM_F32) as p1, plan(M, K, 256) as p2:
        p1.run(dX, dB, dD1)
        p2.run(dY, dZ, dX)          # overwrites X (|values| <= 2 * 256: exact in fp32, rounded once to bf16)
        torch.cuda.synchronize()
        assert p1.sync_status()[0] == dg.GEMM_OK and p2.sync_status()[0] == dg.GEMM_OK
    D1, s1 = ref(X, B)
    r = compare(dD1.double().cpu().numpy(), D1, s1, "f32", 0.0, exact=True)
    assert r["ok"], r
    Xn, _ = ref(Y, Z)
    assert torch.equal(dX.float().cpu(), torch.tensor(Xn).to(torch.bfloat16).float())


def signed_permutation(n, seed):
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(n, generator=g)
    sign = torch.randint(0, 2, (n,), generator=g) * 2 - 1
    w = torch.zeros(n, n)
    w[torch.arange(n), perm] = sign.float()
    return w.to(torch.bfloat16)


def test_chain_of_four_products():
    """T1 = A W1^T, T2 = T1 W2^T, T3 = T2 W3^T, T4 = T3 W4^T with signed
    permutation weights (every intermediate stays in {-2..2}), 64-deep
    contractions, the chain enqueued five times in a row."""
    M, H = 1024, 64
    A = ints((M, H), 21)
    Ws = [signed_permutation(H, 22 + i) for i in range(4)]
    dA = A.cuda()
    dWs = [w.cuda() for w in Ws]
    dT = [torch.empty(M, H, dtype=torch.bfloat16, device="cuda") for _ in range(4)]
    plans = [plan(M, H, H) for _ in range(4)]
    try:
        for _ in range(5):
            src = dA
            for i in range(4):
                plans[i].run(src, dWs[i], dT[i])
                src = dT[i]
        torch.cuda.synchronize()
        for p in plans:
            assert p.sync_status()[0] == dg.GEMM_OK
    finally:
        for p in plans:
            p.close()
    cur = A
    for i in range(4):
        T, _ = ref(cur, Ws[i])
        Tt = torch.tensor(T)
        assert Tt.abs().max() <= 2
        cur = Tt.to(torch.bfloat16)
        assert torch.equal(dT[i].float().cpu(), cur.float()), i
