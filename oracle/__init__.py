"""Plain CPU oracle for the layer-streamed NF4 LoRA path -- TEST INFRASTRUCTURE ONLY.

This package is the slow, obviously-correct reference that the CUDA library is
checked against.  It is written from the pages' statement of the method (and,
for the NF4 code table, from the published NormalFloat construction of the
QLoRA paper), in numpy float64 wherever the pages do not fix a precision; the
NF4 quantisation decision is taken in float32, the precision the kernels use.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import it.  The product package never does, and it shares no
code, table or helper with the CUDA sources.

Sources (by page title and section):

* "Exact Layer Streaming: LoRA Fine-Tuning of an 8B Model on a 4 GB Laptop GPU"
  (abstract): NF4 frozen base + LoRA, layer streaming, bit-exactness of the
  streamed run against a resident run of the same numerics, the cross-entropy
  logits term.
* "Soup CLI Lets You Fine-Tune an 8B LLM on a 4 GB Laptop GPU", sections
  "How Layer Streaming Works" and "v0.73.0: Fixing Silent Wrong Gradients".
* "Soup: Fine-Tuning an 8B LLM on a 4 GB Laptop GPU with One YAML File",
  sections "Layer Streaming: The Mechanism Behind the 4 GB Claim" (pinned base
  store, two device buffers), "The FP32 Bug and What It Means for Your VRAM"
  (base kept in its storage dtype) and "Known Limitations and Failure Modes"
  (adapter gradients must be fp32).

Functions whose parity is not pinned by an independent check say so in their
docstring ("parity unpinned").  At present every function has a pin in
``tests/test_oracle_*.py``.
"""
from . import bf16, nf4, lora, stack, ce  # noqa: F401
