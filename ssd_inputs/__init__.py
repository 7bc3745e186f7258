"""Seeded synthetic inputs for the speculative-decoding verify path.

This module only *generates inputs*: target/draft logits shaped like the
workloads described on the source pages, per-row Philox seeds and fan-out
vectors.  It contains none of the method's arithmetic (no softmax, no
accept test, no sampling from the model distributions); both the CUDA path
and the CPU oracle consume the bytes it produces.

Random draws use numpy's ``Philox`` bit generator keyed by
(workload seed, sequence index), so every sequence of a batch can be
regenerated on its own, bit-for-bit, on any host.

Sources (cited by page title and section):

* [SSD-note] "论文阅读：Speculative Speculative Decoding — 消除推测解码的最后一个顺序瓶颈"
* [SD-7.3]   "7.3 Speculative Decoding：投机采样加速"
* [SD-blog]  "推测解码：用一个“小模型”骗出 3 倍推理速度"
"""

from .generators import (  # noqa: F401
    WORKLOADS,
    Workload,
    bf16_bits,
    bf16_to_f32,
    make_batch,
    sequence_logits,
)
