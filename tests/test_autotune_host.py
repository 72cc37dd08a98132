"""The autotuner's host logic on CPU: which plans it would time for a shape
(every family the library can run it with, no others) and its shape syntax."""
from dense_gemm_11_gb300 import GEMM_PATH_F32, GEMM_PATH_TC, autotune


def test_fp32_candidates():
    c = autotune.candidates(GEMM_PATH_F32, 512, 512, 512)
    assert (1, 0, 0) in c  # big persistent tiles
    splits = sorted(s for v, _, s in c if v == 2)
    assert splits[0] == 1 and splits[-1] <= 512 // 32 // 2  # 64x64 tiles, at most half the k slices
    assert all(v in (1, 2) and bn == 0 for v, bn, _ in c)


def test_tensor_core_candidates_by_family():
    # large M: pairs and single-CTA tiles, no transposed small-M family
    c = autotune.candidates(GEMM_PATH_TC, 4096, 4096, 4096)
    fams = {v for v, _, _ in c}
    assert {1, 2} <= fams and 3 not in fams
    assert {bn for v, bn, _ in c if v == 1} == {256, 224, 192}
    # cluster split (variant 4) only where tiles x splits fit on the SMs
    c = autotune.candidates(GEMM_PATH_TC, 128, 4096, 4096)
    v4 = [(bn, s) for v, bn, s in c if v == 4]
    assert v4 and all(2 <= s <= 8 for _, s in v4)
    assert all(((4096 + bn - 1) // bn) * s <= autotune.sm_count() for bn, s in v4)
    # small M adds the transposed family, with MMA N at least M
    c = autotune.candidates(GEMM_PATH_TC, 48, 4096, 4096)
    assert {bn for v, bn, _ in c if v == 3} == {64}
    c = autotune.candidates(GEMM_PATH_TC, 16, 4096, 4096)
    assert {bn for v, bn, _ in c if v == 3} == {32, 64}
    # one k block: nothing to split
    c = autotune.candidates(GEMM_PATH_TC, 16, 4096, 64)
    assert all(s <= 1 for v, _, s in c if v in (2, 3)) and not [1 for v, _, _ in c if v == 4]


def test_shape_syntax():
    assert autotune._parse_shape("tc:128x11008x4096") == (GEMM_PATH_TC, 128, 11008, 4096)
    assert autotune._parse_shape("f32:512X512x512") == (GEMM_PATH_F32, 512, 512, 512)
