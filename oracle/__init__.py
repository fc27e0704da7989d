"""CPU oracle for NVFP4 fake-quantized attention training (Attn-QAT).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or link
this package: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` use it.  It shares no code, table or constant generator with
the CUDA library under ``nvfp4_fake_quant_gb300/csrc``.

Modules
-------
``nvfp4``      the NVFP4 block quantizer (E4M3 scale per 16 elements, E2M1 codes),
               in numpy with an explicit arithmetic precision, plus an exact
               ``fractions.Fraction`` version used to pin it.
``attention``  forward and straight-through backward of fake-quantized attention
               in float64, whole-tensor and sampled (per query row / per key),
               dense or block-sparse (a list of key tiles per query tile).
``vsa``        video sparse attention: cube token order, the top-k formula and
               the cube-mean score selection of key tiles.
``linear``     the NVFP4 linear: quantized forward with the FP4 GEMM's global-scale
               alpha, straight-through backward, the 128 x 4 tiled scale layout.

Sources (web pages on the subject; cited by title and section):
  * "nvfp4_qad.py" (FastVideo ``fastvideo/layers/quantization/nvfp4_qad.py``):
    module docstring (NVFP4 format, unit and static global scale, STE with a
    full-precision backward), ``weight_global_sf`` (448*6/amax, fp32, clamp),
    ``nvfp4_gemm`` (alpha = (1/w_sf)/input_sf, i.e. value = code*scale/gsf).
  * "attn_qat_train" API page: the source of ``attn_qat_train()`` (which of
    Q, K, V and P are quantized, unit global scales, STE backward flags,
    default softmax scale 1/sqrt(D)).
  * "Attn-QAT Training" guide, section "Architecture-specific Triton routing"
    (the exact-m statistics switch).
  * "vsqa-preview-1.3b metadata.json", ``attention.precision`` of the dense
    ATTN_QAT_TRAIN ancestor (group size 16, NVFP4 E2M1 values, FP8 E4M3FN
    scales, quant_p, quant_v, no two-level P, backward "consistent STE"), and
    ``attention`` of the VSA run (cube_shape, selection sparsity and top-k).

Every function is pinned by ``tests/test_oracle_*.py`` (hand-worked examples,
library routines, brute force, invariants); none is marked "parity unpinned".
"""
