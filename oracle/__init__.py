"""Plain fp64 CPU oracle for video-DiT attention (test infrastructure only).

This package is the correctness reference that the CUDA path is checked against. It is
slow on purpose and written so each step can be read against its source passage:

* ``rope``      -- split-halves rotary embedding, 1-D and 3-D (t, h, w) angle tables.
* ``attention`` -- softmax(q~ k~^T * scale) v with explicit pad-key masking, the natural-log
                   LSE, sampled-row evaluation for large inputs, and the LSE merge of
                   partial results over key shards.
* ``brute``     -- a pure-Python per-query loop (math.fsum) used to pin the numpy oracle on
                   tiny inputs.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may import
this package. The product path (``video_dit_attention_gb300``) never imports it, and the
two share no code: only the seeded input generators in ``video_dit_attention_gb300.inputs``
feed both sides.

Pinning status (what fixes each function other than itself; the pins live in
``tests/test_oracle_*.py`` and ``tests/golden/``):

* attention core, masking, LSE: brute force, closed forms (q = 0, one valid key),
  torch's fp64 scaled_dot_product_attention and logsumexp, permutation invariance,
  pad-content invariance.
* split-halves rotation: complex-multiply form, norm preservation, identity at position 0,
  relative-position property, equivalence with interleaved rotary under the channel
  permutation the Difflet page applies to q/k.
* LSE merge: sharded-then-merged equals unsharded; one shard is the identity; an empty shard
  contributes nothing; an independent log-sum-exp.
* 3-D axis-to-channel assignment (pairs 0-21 -> t, 22-42 -> h, 43-63 -> w) and the rotation
  sign: parity unpinned -- the pages print no worked example, so these follow the stated
  reading only (the per-axis relative-position property still holds and is tested).
"""
