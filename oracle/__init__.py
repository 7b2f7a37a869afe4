"""Plain CPU oracle for the microscaled (OCP MX) quantized linear layer.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may use it.  It shares no code,
table or constant generator with the CUDA library, and it never reads a value
produced by the CUDA library.

Every function computes what the source pages define, in fp64 (or exactly, with
integer arithmetic), with no blocking, fusion or reordering beyond the
definition.  Sources, cited by page title and section:

* ``weights942``  = vllm.models.deepseek_v41.amd.mono.weights942
  (sections: ocp_from_dequant, dense_copy, fp4_drop_negative_zero_,
  linear_copy, moe_copies, fp4_lane_major)
* ``rocm_native`` = vllm.model_executor.kernels.linear.mxfp8.rocm_native
  (sections: _quant_mxfp8_tile, _launch, apply_weights,
  process_weights_after_loading, _as_block32_scale)
* ``a16w4``       = vllm.models.minimax_m3.amd.specialized_decode.mono.a16w4
  (sections: module text, dequant, scale_f32)

Modules:

* ``formats``  e4m3 / e2m1 / E8M0 / bf16 decode and round-to-nearest-even encode
* ``quant``    per-token MXFP8 activation quantizer
* ``layout``   the library's packed weight layout as plain index maps (+ inverse)
* ``linear``   MXFP8 x MXFP8 linear and dequant, fp64
* ``moe``      token->expert routing and the A16W4 expert linear, fp64

Parity status of each function is stated in its docstring ("pinned by ..." or
"parity unpinned").
"""
