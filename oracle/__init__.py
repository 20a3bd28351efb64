"""CPU fp64 oracle for the partitioned-attention hot path.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, obviously correct
restatement of what the hot path computes, written from the pages that define
the method.  Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline / reference legs may import it.  The CUDA library and its Python
binding never import, call or link anything here, and nothing here imports the
CUDA path: the two share no code.  The only shared module is the seeded input
generator ``partitioned_kv_cache_gb300.workload``, which holds none of the
method's arithmetic.

Sources (cited by title and section throughout):

* "Reflex: Real-Time VLA Control through Streaming Inference" (paper review
  page) -- §III "Core formulas": Eq. (1) partitioned attention, Eq. (2)
  AdaRMSNorm, Proposition A.1; §III "System architecture" (ring-buffer
  partitions, FIFO of N observations); §III "Model components" (ring buffer,
  AdaRMSNorm MLP); §V "Key implementation" (StreamingInputManager methods,
  ring-buffer initialisation, AdaRMSNorm forward).
* "OxyGen: Unified KV Cache Management for Vision-Language-Action Models under
  Multi-Task Parallelism" (summary page) -- §"Core method" (cross-task KV
  sharing: read-only action view, language streams appending private KV).

Modules:

* ``ring``      -- logical FIFO window of frames (pinned / sliding regions).
* ``attention`` -- Eq. (1) over explicitly concatenated K/V; region-split
                   evaluation for Proposition A.1; pure-Python brute force.
* ``adarms``    -- sinusoidal timestep embedding, gamma MLP, Eq. (2).
* ``pipeline``  -- one stream tick of the hot path built from the above.

Every function is pinned by ``tests/test_oracle_*.py`` against closed forms,
invariants, brute force or an independent library routine.
"""
