"""CPU oracle for the CSA2 global-attention hot path -- TEST INFRASTRUCTURE ONLY.

Plain, slow, float64 NumPy restatement of what the path computes, written from
the four source pages (cited by page title and section in each function):

  [P1] "DeepSeek-V4.1 模型结构（2）：序列维度（中），CSA2 的三种模式" (blog.javazero.top)
  [P2] "DeepSeek v4.1 Flash技术剖析——架构篇" (myhz0606.com)
  [P3] "DeepSeek-V4.1-Flash：把百万 Token 的记忆，压缩成一套分级缓存" (junki.cn)
  [P4] "CSA2 — l'attention creuse compressée de seconde génération" (mkdocs.reaper.mx)

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA library
(``compressed_sparse_attention_04_gb300``) and imports nothing from it; the
only module both sides use is the seeded input generator ``synth``.

Parity-unpinned readings (the pages print no value that could confirm them):
RMSNorm epsilon 1e-6; interleaved RoPE pairs; the ReLU form of the indexer
score; the E4M3 scale rule amax/6 rounded to nearest-even; FP4 quantisation of
indexer queries; the attention-sink form; the 1/sqrt(512) attention scale;
the stored formats' group sizes (FP4 main KV: one E4M3 scale per 16 channels;
FP8 window rows: one power-of-two scale per 64 channels, ``fp8.py``).
Each is a single named constant or switch in ``csa2_ref`` / ``fp8``.
"""
