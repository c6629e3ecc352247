"""CPU oracle for the tensor-parallel linear layer and its flat param/grad buffer.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the ``param_buffers_gb300``
package, its CUDA library, the C ABI) imports, links or executes anything here.  The
only callers are ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py``.

The oracle is plain and slow on purpose: float64 NumPy, integer bit arithmetic for the
number formats, pure-Python loops for the tiny brute-force cases.  It shares no code,
tables or constants with the CUDA path.

Pages the oracle follows (cited by short tag throughout):

* [LIN] "01 · ColumnParallelLinear / RowParallelLinear and the core autograd"
  (llm-infra-atlas, parallel/02_tp_sp) - the fprop / dgrad / wgrad GEMMs, §4.1, §4.2.
* [BUF] "05 · grad/param buffer: contiguous buffer data structures and read/write loop"
  (llm-infra-atlas, train/05) - BufferKey §3, layout §4.1-§4.3, mounting §5,
  the run-time loop §6.3/§6.5/§6.6, the memory ledger §8.
* [MLM] "Megatron-LM architecture and source guide" (arganzheng.life) - parameter
  counts §1 (overview), run.sh §4, DDP buffers §6.3, DistributedOptimizer §6.4.
* [GTP] "Generalized Tensor Parallelism (GTP)" (Megatron-Core developer guide) -
  MXFP8 block-32 weights, §1.3 and its "Communication volume breakdown" table.

Modules:
  llama_shapes  parameter counts of the Llama-3.2-1B shape            (pinned)
  layout        BufferKey grouping, reverse placement, padding, cuts   (pinned)
  gemm          fprop / dgrad / wgrad-accumulate definitions           (pinned)
  floats        bf16 and E4M3 round-to-nearest-even, E8M0 scales       (pinned)
  adamw         AdamW on fp32 master/m/v, the fused buffer sweep       (pinned)
  mxfp8         MX block quantize (block 32) and the MXFP8 fprop        (pinned)
  gradnorm      per-bucket sums of squares, norm and clip coefficient  (pinned)
  nvfp4         NVFP4 quantize (block 16, tensor scale) and its fprop  (pinned)
  sf_layout     the tiled order of scale bytes                         (pinned)
  rs_sum        the local fp32 sum of the all-to-all reduce-scatter    (pinned)

Every function is pinned by a ``-m "not gpu"`` test against something other than
itself (page-printed values under tests/golden/, closed forms, library special cases,
brute force).  The one value the pages print that cannot be reproduced (the toy's
``param_data sum``) is listed as "parity unpinned" in the layout module.
"""
