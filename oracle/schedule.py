"""Max-plus pipeline schedule of a warp-specialised GEMM main loop.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).  Plain Python in the
notation of "Hopper and Blackwell GEMM", section "Maths": K slices numbered
g = t*K + k (tile t, slice k), S stages, A accumulator buffers, and

    L_g = max(L_{g-1} + t_issue, D_{g-S})
    M_g = max(L_g + t_load, D_{g-1}, E_{t-A} if k = 0)
    D_g = M_g + t_mma
    E_t = max(D_{tK+K-1}, E_{t-1}) + t_epi

Terms whose index is negative are absent; the first issue is at time 0.

parity pins: tests/test_schedule.py (the page's printed busy fractions and run
lengths, its closed form and steady-state equation).
"""


def model(T, K, S, A, t_issue, t_load, t_mma, t_epi):
    L, M, D, E = {}, {}, {}, {}
    for t in range(T):
        for k in range(K):
            g = t * K + k
            candidates = [L[g - 1] + t_issue] if g >= 1 else [0.0]
            if g - S >= 0:
                candidates.append(D[g - S])
            L[g] = max(candidates)
            candidates = [L[g] + t_load]
            if g - 1 >= 0:
                candidates.append(D[g - 1])
            if k == 0 and t - A >= 0:
                candidates.append(E[t - A])
            M[g] = max(candidates)
            D[g] = M[g] + t_mma
        candidates = [D[t * K + K - 1]]
        if t - 1 >= 0:
            candidates.append(E[t - 1])
        E[t] = max(candidates) + t_epi
    run = E[T - 1]
    return {"L": L, "M": M, "D": D, "E": E, "run": run, "busy": T * K * t_mma / run}
