"""CPU oracle for the sparse-decode hot path -- TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously correct fp64 numpy restatements of what each step of the
path computes.  Only the test-suite, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it; the
library's product path never does, and it shares no code with the CUDA kernels.

Sources (pages about the SparseEngine sparse-first inference engine):

* "tokendh.com article" -- the tokendh.com news article on SparseEngine;
  sections "历史太长,会撑爆什么" (the four method families; Quest picks pages by
  query, H2O keeps a running accumulated attention score and deletes),
  "把边界划在'生命周期'上" (SnapKV looks at the last few tokens' attention over
  the history and physically deletes the rest; H2O updates its scores every
  decode step then decides what to delete; AttentionView turns each method's
  cache into one format the attention reads).
* "SparseEngine 统一接入十五种稀疏注意力" -- the Netics blog page, section
  "SparseEngine 围绕 KV cache 构建了什么".
* "SparseEngine：稀疏优先推理引擎" -- the ai-feeds.com paper card, section
  "方法 / 关键模块" (AttentionView exposes the selected positions uniformly).
* "长程 agent 把显存撑爆以后" -- the jetabc.cn explainer, section
  "四、为什么进不了 vLLM 一类的引擎" (fixed-size KV pages plus a table that
  maps each token to its page).

The pages print no formulas.  The operations are the textbook definitions of
Quest, SnapKV and H2O as this library specifies them (each function states
its definition); every reading of a point the pages leave open is named in
the function that takes it.

Parity pins: every function here is pinned by tests under ``tests/`` marked
``not gpu`` (closed forms, invariants, brute force, library routines).
"""

from .bf16 import widen  # noqa: F401
from .topk import rank_order, top_k  # noqa: F401
from .quest import page_minmax, quest_bound, quest_bound_max, quest_k_pages, quest_select  # noqa: F401
from .attention import attend, logits  # noqa: F401
from .snapkv import window_scores, max_pool, keep_positions, compact  # noqa: F401
from .h2o import H2OState, h2o_init, h2o_step  # noqa: F401
from .omnikv import omnikv_layers, source_layer, filter_pages  # noqa: F401
from .prune import span_keep_positions, sink_recent_pages  # noqa: F401
