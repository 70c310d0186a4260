"""GDPA oracle.  TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct CPU implementation of what the GDPA hot path
computes, used to check the CUDA library.  Only the tests, the smoke check and
the CPU-baseline leg of the benchmark may import it; the library itself never
does, and this package imports nothing from the library.

* ``ref``     float64 C loops (forward, backward, activations), via ctypes;
              also the softmax variant (Jagged Flash Attention, forward).
* ``brute``   dense padded NumPy float64 formulation of the same maths.
* ``planner`` the host tile plan (valid tiles, costs, zigzag / round-robin
              dealing) restated in plain Python.
* ``mx``      MXFP8 quantisation (E4M3 elements, E8M0 scales per 32 values)
              in float64, for the block-scaled variant.
* ``rmsnorm`` the RMSNorm prologue on Q and K and its gradient, composed
              with the GDPA loops.

The method follows the GDPA page ("범용 내적 어텐션(GDPA): 실제 추천 시스템
학습 부하를 위한 커널 최적화", aitrends.kr): its summary and first detailed
section for the formula, the scheduling paragraph and diagram for the planner,
and the Taylor GELU code figure for the polynomial activation.  The softmax
variant is the Jagged Flash Attention kernel the GEM page ("GEM 트레이닝:
Meta가 LLM 규모의 광고 파운데이션 모델 효율성을 두 배로 높인 방법",
techlist.io, section "GPU 연산 효율을 높인 맞춤형 커널과 정밀도") lists beside
GDPA.
"""

ACT_IDS = {"gelu_erf": 0, "gelu_tanh": 1, "silu": 2, "gelu_taylor6": 3, "identity": 4,
           "softmax": 5}
MASK_IDS = {"none": 0, "causal_window": 1}
