"""Float64 CPU oracle for the NVFP4-KV decode-attention path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this package: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` use it.  It shares no code with the CUDA path
(``precision_kv_cache_gb300``); the two meet only at the seeded inputs of
``workloads``.

It is written to be read against its sources, not to be fast:

* ``formats``  - E2M1 / E4M3 value tables and the NVFP4 / FP8 encoders, from
  the OCP Microscaling (MX) v1.0 and OCP 8-bit floating point definitions and
  the rounding contract of this library (nearest, ties to the even code,
  saturate to the largest finite value).
* ``layout``   - where each code and scale byte of a token lives in a 64-token
  page of the cache (a definition of this library, written out byte by byte).
* ``attention`` - softmax attention over the dequantized global cache plus the
  FP8 sliding window (decode), the bounded replay of the last 128 tokens after
  a prefix hit, the log-sum-exp merge of partial results, the sparse index
  score sum_h w_h*ReLU(q_h . k_t) and its top-k, all in float64.

Sources (page title, section):
[blog]  "DeepSeek-V4.1-Flash sur vLLM : 5x de débit agentique dès le jour 0"
        (spke.com, French translation of the vLLM blog) - sections
        "SWA bounded replay", "Côté encodeur : reconstruire la fenêtre lors
        d'un hit de cache", "Kernels" (paragraphs "Logits MQA creux",
        "MegaAttention avec KV compressé NVFP4"), "Performances agentiques".
[news]  cocoloop news summary of the same blog (fr/de/pt/es), section
        "Les particularités du modèle lui-même".

Parity status: every function here is pinned by tests that do not reuse its
code (literal OCP tables, worked examples, closed forms, brute force with
``math.fsum`` on tiny inputs, a second formulation of the rotary embedding by
complex multiplication).  The sources print no worked example of an
attention output at the bench sizes; what fixes those values is the pinned
definition, which holds at any size.
"""
from . import formats, layout, attention  # noqa: F401
