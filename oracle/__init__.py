"""Oracle for displaced patch parallelism: a plain, slow fp64 CPU statement.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or
links this package; only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use it.  It shares no code, table or helper
with the CUDA library.

Sources, cited in the docstrings by the short tag in brackets:

[DF-notes]  "阅读论文1_b" -- reader's notes on "DistriFusion: Distributed
            Parallel Inference for High-Resolution Diffusion Models"
            (Introduction para. 3-5; Related Work / Parallelism; Background).
[DF-guide]  "DistriFusion开发者必读：分布式UNet架构设计与模块拆分实现详解"
            (sections 卷积层拆分 convolution split, 注意力机制拆分 attention
            split, 归一化层拆分 normalisation split, 分布式通信与同步机制
            communication and synchronisation).
[Hydiff-zh] gist.science summary of "Hybridiff / Hydiff" (arXiv 2602.21760),
            sections "基于条件的数据划分" (condition-based partitioning) and
            "自适应并行切换" (adaptive parallelism switching).
[Hydiff-ru] Denis Avetisyan, "Ускорение генерации изображений: новый подход к
            параллельным вычислениям", section "Адаптивное переключение"
            (denoising discrepancy).

The one definition everything below follows.  An image of H rows is cut into
P horizontal bands (the gathered buffer is rebuilt by concatenation along the
height axis, [DF-guide] communication section); band p owns rows
R_p = [p*H/P, (p+1)*H/P).  At a displaced step, device p computes its own rows
from fresh activations F and takes the other bands' activations from the
previous step, the stale buffer S ([DF-notes] Introduction para. 4; Related
Work / Parallelism).  So each displaced layer is the ordinary full-image layer
applied to the composite image Z_p (F on R_p, S elsewhere), kept on R_p.
The first step is synchronous: S == F ([DF-notes] Introduction para. 4).

Pins: see tests/test_oracle_pins.py.  Every function here is checked there
against something other than itself (torch library routines on the special
cases S == F and P == 1, brute-force loops on tiny inputs, closed forms and
invariants).
"""
from .displaced import (  # noqa: F401
    patch_rows,
    patch_of_row,
    composite,
    conv3x3,
    displaced_conv3x3,
    naive_conv3x3,
    groupnorm,
    groupnorm_partials,
    displaced_groupnorm,
    naive_groupnorm,
    attention_heads,
    linear,
    kv_state,
    displaced_self_attention,
    naive_self_attention,
    cross_attention,
    cfg_combine,
    rel_mae,
    refresh_stale,
    switch_stages,
    WARMUP,
    PARALLEL,
    FULLY_CONNECTING,
)
