"""CPU oracle of the NVFP4 W4A4 Gated DeltaNet layer step.

TEST INFRASTRUCTURE, NOT PRODUCT CODE. Only the test suite, the package's
smoke check and the benchmark's CPU-baseline leg may import or call anything
here. The CUDA path never imports it, and it never imports the CUDA path: the
two share no code, constants or helpers. The only code both sides see is the
seeded input generator (``nvfp4_gated_deltanet_gb300.synth``), which holds none
of the layer's arithmetic.

The oracle is plain and slow on purpose. It computes in float64 (and exact
int64 for the block-scaled dot products) except where the layer fixes a
narrower precision: the NVFP4 quantiser takes its decisions in FP32 (the
precision the kernel decides in), projections are stored in BF16, the
recurrent state is stored in FP32.

What it follows, by page:

* Rocket blog, "A reduction barrier makes Qwen GDN graph replay bit exact",
  setup table: the serving path of one GDN layer is W4A4 QKVZ/BA and output
  projections, a BF16 causal convolution and an FP32 recurrent state; the
  recurrence follows vLLM's fused_recurrent gated delta rule, the decode state
  layout follows FlashInfer's "pretranspose" decode (state stored [v][k]).
* bloomery issue #565, §4 (#489/#687): NVFP4 is U8-packed E2M1 pairs with
  one F8_E4M3 scale per 16 values and an FP32 per-tensor scale; W4A4 means the
  activations are quantised to NVFP4 too.
* Rocket blog, "Moving the KDA state tile out of shared memory is 4.6x at M=8",
  Correctness: a double-precision evaluation of the recurrence is the
  reference and tolerances are relative.

Every stage whose exact form the pages leave open takes the reading written in
its docstring.
"""
from . import codecs, nvfp4, gdn, fnv  # noqa: F401
