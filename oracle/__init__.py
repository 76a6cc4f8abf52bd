"""CPU oracle for the Introspective Strided Decoding (ISD) verify/accept step.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code with the CUDA library (``speculative_verify_accept_step_b300``) and
neither side imports the other.

Everything here is plain NumPy in float64: slow, written to be read against the
pages it cites.  The pages are four web pages about Introspective Diffusion
Language Models (I-DLM); they are cited by title and section:

* [IDLM] "Introspective Diffusion Language Models" -- the project page
  (news.routley.io/posts/introspective-diffusion-language-models.html):
  sections "Inference & ISD", "Serving (SGLang)", "Lossless R-ISD",
  "Training", "How do DLMs perform as they approach compute-bound?" and the
  speedup panel ("I-DLM acceptance rate (p)", "Memory-bound: Speedup ~ TPF").
* [GN] "I-DLM - Icgozlemsel Difuzyon Dil Modelleri (Introspective Diffusion
  Language Models)" -- GeekNews summary (tr.news.hada.io/topic?id=28562):
  sections "I-DLM Yontemi", "Throughput", "Speedup Factor Explorer",
  "Inference & ISD", "Serving (SGLang)", "Lossless R-ISD".
* [ABS] "Modelos de Lenguaje de Difusion Introspectiva" -- the paper abstract
  (chatpaper.ai), English paragraph.
* [OJ] ojeo.com news note on I-DLM ("modelos de lenguaje: nueva tecnica
  supera limitaciones").

Modules:
  philox    Philox4x64-10 counter-based generator (Salmon et al., SC'11) and the
            uniforms the accept step draws.
  isd       attention, accept (p/q rule, residual resample, proposals), KV
            commit, gated LoRA, the TPF closed form and a decode loop.

Parity pins live in ``tests/test_oracle_*.py``.  One function is marked
"parity unpinned" in its docstring: the ARGMAX-proposal acceptance numbers
(no page gives a value to compare against).
"""

from . import philox, isd  # noqa: F401
