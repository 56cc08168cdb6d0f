"""Host-side launch planning (w4a16_launch_plan; no GPU): for a grid of layer
shapes, SM counts and paths, the plan each kernel would launch with keeps the
kernels' constraints - the K split divides the work into CTAs that each keep
whole K boxes, the small-M kernel's ring fits shared memory, a split
tensor-memory launch fits on the GPU at once, the tiles cover M and N exactly -
and AUTO follows the router's measured crossovers."""

import itertools

import pytest

from w4a16_int4_weight_gb300 import build as wbuild


@pytest.fixture(scope="module")
def B():
    wbuild.build()
    from w4a16_int4_weight_gb300 import binding
    return binding


def cdiv(a, b):
    return -(-a // b)


MS = [1, 2, 3, 5, 8, 9, 13, 16, 17, 31, 32, 33, 64, 65, 100, 128, 129, 256, 300, 1000, 2048, 4096]
NS = [8, 128, 136, 1024, 4096, 11008, 14336, 28672]
KS = [16, 48, 256, 272, 1024, 4096, 8192, 11008, 14336]
GS = [-1, 32, 64, 128, 256]


def valid(N, K, G, qt):
    ge = K if G == -1 else G
    return K % 16 == 0 and K % ge == 0 and (qt == "uint4b8" or N % 8 == 0)


def shapes():
    for N, K, G, qt in itertools.product(NS, KS, GS, ["uint4b8", "uint4"]):
        if valid(N, K, G, qt):
            yield N, K, G, qt


def check_decode(p, M, N, K):
    nboxes = cdiv(K, 256)
    assert p["k_split"] in (1, 2, 4, 8) and p["k_split"] <= nboxes
    per_cta = cdiv(nboxes, p["k_split"])
    assert 1 <= p["stages"] <= 5 and (p["stages"] == 1 or p["stages"] <= per_cta)
    nt = next(t for t in (1, 2, 4, 8) if 8 * t >= M)
    assert p["token_tile"] == 8 * nt
    assert p["grid"] == cdiv(N, 128) * p["k_split"]
    # each ring stage holds a 16 KB packed weight box and the [M x 256] activation box
    assert p["stages"] * (16384 + M * 512) <= p["smem_bytes"] <= 227 * 1024


def check_tmem(p, M, N, K, sms):
    tt = next((t for t in (16, 32, 64) if t >= M), 128)
    assert p["token_tile"] == tt
    ks = p["k_split"]
    assert ks in (1, 2, 4, 8)
    tiles = cdiv(N, 128) * cdiv(M, tt)
    if ks > 1:
        assert cdiv(K, 256) // ks >= 2            # every CTA keeps at least two weight stages
        assert p["grid"] <= 2 * sms              # all CTAs of the split launch fit at once
    if ks == 2 and p["grid"] != tiles * ks:
        # between one and two 32- or 64-token tiles per SM: clusters of two take two
        # whole tiles or split one, exactly two CTAs per SM
        assert tt in (32, 64) and sms < tiles < 2 * sms, (M, N, K, sms)
        assert p["grid"] == 2 * sms
    else:
        assert p["grid"] == tiles * ks
    assert p["stages"] == 0 and p["smem_bytes"] == 0


def test_plans_keep_the_kernel_constraints(B):
    n = 0
    for (N, K, G, qt), M, dt, sms in itertools.product(list(shapes()), MS, ["bf16", "fp16"], [148, 152]):
        for has_dense in (False, True):
            auto = B.launch_plan(M, N, K, G, qt, dt, "auto", has_dense, sms)
            routed = B.lib.w4a16_route(M, N, K, G, B._qt(qt), B._dt(dt), int(has_dense))
            assert auto["path"] == B.PATH_NAMES[routed]
            # the router's crossovers (measured): small M on the split-K kernel, except
            # 9..16 tokens at 32-wide groups with zero points below 2^27 weights; the
            # dense copy from 2048 tokens
            g32 = G == 32 and K > 32 and qt == "uint4" and N * K < 2 ** 27
            if M <= 8 or (M <= 16 and not g32):
                assert auto["path"] == "decode", (M, N, K, G)
            elif has_dense and M >= 2048:
                assert auto["path"] == "dense"
            else:
                assert auto["path"] == "fused_tmem"
        if M <= 64:
            check_decode(B.launch_plan(M, N, K, G, qt, dt, "decode", False, sms), M, N, K)
        check_tmem(B.launch_plan(M, N, K, G, qt, dt, "fused_tmem", False, sms), M, N, K, sms)
        ps = B.launch_plan(M, N, K, G, qt, dt, "fused_smem", False, sms)
        tt = 64 if M <= 64 else 128 if M <= 128 else 256
        assert ps["token_tile"] == tt and ps["k_split"] == 1
        assert ps["grid"] == cdiv(N, 128) * cdiv(M, tt)
        pd = B.launch_plan(M, N, K, G, qt, dt, "dense", False, sms)
        assert pd["token_tile"] == 256 and pd["k_split"] == 1
        assert pd["grid"] == min(sms, cdiv(N, 128) * cdiv(M, 256))
        n += 1
    assert n > 10000


def test_fused_mixed_clusters_between_one_and_two_tiles_per_sm(B):
    # 224 row tiles of 32 tokens: whole tiles would leave SMs unevenly loaded, so
    # clusters of two take two whole tiles or split one, two CTAs on every SM
    for sms in (148, 152, 200):
        p = B.launch_plan(32, 28672, 8192, 64, "uint4b8", "bf16", "fused_tmem", False, sms)
        assert (p["token_tile"], p["k_split"], p["grid"]) == (32, 2, 2 * sms)
    # one tile per SM or fewer: the plain split; two or more: whole tiles
    p = B.launch_plan(32, 28672, 8192, 64, "uint4b8", "bf16", "fused_tmem", False, 224)
    assert (p["k_split"], p["grid"]) == (2, 448)
    p = B.launch_plan(32, 28672, 8192, 64, "uint4b8", "bf16", "fused_tmem", False, 100)
    assert (p["k_split"], p["grid"]) == (1, 224)
    # the same at 64-token tiles (their split CTAs reduce through the activation ring)
    p = B.launch_plan(64, 28672, 8192, 64, "uint4b8", "bf16", "fused_tmem", False, 152)
    assert (p["k_split"], p["grid"]) == (2, 304)
    # 128-token tiles keep whole tiles
    p = B.launch_plan(128, 28672, 8192, 64, "uint4b8", "bf16", "fused_tmem", False, 152)
    assert (p["k_split"], p["grid"]) == (1, 224)


def test_route_does_not_depend_on_the_sm_count(B):
    # w4a16_route takes no SM count: the path AUTO resolves to must be the same
    # whatever SM count a launch is planned for, and the small-M plan must exist
    # for every count whenever the router picks it
    n = 0
    for (N, K, G, qt), M in itertools.product(list(shapes())[::7], [1, 4, 9, 16, 17, 64]):
        for dt in ("bf16", "fp16"):
            want = B.route(M, N, K, G, qt, dt)
            names = {v: k for k, v in B.PATHS.items()}
            for sms in (1, 2, 7, 64, 132, 148, 152, 160, 1000, 4096):
                p = B.launch_plan(M, N, K, G, qt, dt, "auto", False, sms)
                assert p["path"] == names[want], (M, N, K, G, qt, dt, sms)
                if p["path"] == "decode":
                    check_decode(p, M, N, K)
                n += 1
    assert n > 1000


def test_plans_of_the_measured_workloads(B):
    # the launches the ncu summaries were taken on
    p = B.launch_plan(8, 4096, 4096, 128, "uint4b8", "bf16")
    assert (p["path"], p["k_split"], p["stages"], p["grid"]) == ("decode", 8, 2, 256)
    p = B.launch_plan(1, 28672, 8192, 64, "uint4b8", "bf16")
    assert (p["path"], p["k_split"], p["stages"], p["grid"]) == ("decode", 2, 4, 448)
    p = B.launch_plan(2048, 14336, 4096, 128, "uint4b8", "bf16")
    assert (p["path"], p["token_tile"], p["k_split"], p["grid"]) == ("fused_tmem", 128, 1, 1792)
    p = B.launch_plan(2048, 14336, 4096, 128, "uint4b8", "bf16", has_dense=True)
    assert (p["path"], p["grid"]) == ("dense", 152)


@pytest.mark.parametrize("args,needle", [
    ((0, 4096, 4096, 128, "uint4b8", "bf16"), "M="),
    ((1, 4096, 4100, 128, "uint4b8", "bf16"), "K"),
    ((1, 4096, 4096, 7, "uint4b8", "bf16"), "group size"),
    ((1, 4100, 4096, 128, "uint4", "bf16"), "N"),
])
def test_plan_rejects_what_the_gemm_rejects(B, args, needle):
    with pytest.raises(B.W4A16Error, match=needle):
        B.launch_plan(*args)


def test_plan_rejects_bad_path_and_sm_count(B):
    with pytest.raises(B.W4A16Error, match="num_sms"):
        B.launch_plan(1, 4096, 4096, 128, "uint4b8", "bf16", num_sms=0)
    with pytest.raises(B.W4A16Error, match="unknown path"):
        B.launch_plan(1, 4096, 4096, 128, "uint4b8", "bf16", path=9)
    with pytest.raises(B.W4A16Error, match="decode path takes"):
        B.launch_plan(65, 4096, 4096, 128, "uint4b8", "bf16", path="decode")
