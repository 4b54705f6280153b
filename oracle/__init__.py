"""CPU oracle of the shared quantized KV pool.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports, links or runs
this package: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU legs of
``bench.py`` (``cpu_baseline`` and ``--impl reference``) may use it. It shares
no code with the CUDA library; both sides consume the same seeded input bytes
from ``shared_quantized_kv_gb300.workloads``, which holds no arithmetic of the
method.

What it computes (a plain restatement of the pages, slow and in plain numpy):

* ``lloyd_max``  -- the Lloyd-Max scalar quantiser for N(0, 1) with 4, 8 and 16
  levels (float64), and its float32 centroid / midpoint tables.
* ``codec``      -- the write-once encode of one layer: per-tensor symmetric int8
  K, and V rotated per head-vector by the fast Walsh-Hadamard transform, scaled
  to N(0, 1) by the vector norm and mapped to the nearest centroid, bit-packed;
  and the decompress (centroid lookup + inverse FWHT) to bf16; layers built
  from 32-token groups of their own V widths (``encode_layer_groups``).
* ``attention``  -- float64 decode attention of every agent's query rows over
  the dequantised pool plus the agent's private bf16 tail (plain softmax
  definition).

Sources, cited by page title and section:

* "PolyKV: A Shared Asymmetrically-Compressed KV Cache Pool for Multi-Agent LLM
  Inference" (gist.science summary), section 2.A (SharedKVPool, PooledAgent) and
  2.B (asymmetric compression: int8 K per tensor; V by FWHT rotation + Lloyd-Max
  N(0,1) centroids, 3-bit; dequantisation by centroid lookup + inverse FWHT;
  ratio 16/((8+3)/2)).
* "CoMixKV ... Qwen3显存降低32.08%" (zicq.com article), sections on the
  incremental quantisation strategy (recent states stay at native precision;
  a new width applies only to blocks quantised afterwards) and on 2-4 bit
  per-layer precision.

Where the pages are silent the readings are fixed in each function's docstring.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against closed forms, published tables (Max 1960), exact rational arithmetic on
tiny inputs, or brute force. None is "parity unpinned".
"""

from . import lloyd_max, codec, attention  # noqa: F401
