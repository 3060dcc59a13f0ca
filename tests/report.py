"""Quantities the GPU tests measure and print at the end of the run (no
heavy imports: conftest reads it in every session)."""

# (config, rows, relative L2 error, max |error|, max |Y_exact|) of the layer's
# fp16 Y against the unquantized fp64 product X W^T (+ the LoRA term).
QUANT_ERRORS = []
