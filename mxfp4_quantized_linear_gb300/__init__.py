"""MX (MXFP8 / MXFP4) quantized linear for one GB300 (sm_103a)."""
