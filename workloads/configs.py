"""The five synthetic decode workloads and a generic spec for test cases.

Shapes follow the generation-phase decode problem described on the XQA page
("TensorRT-LLM 源码完全拆解(二十九)", section on decode constraints), the MetaX
grouped kernel PR (performance table: 32/4 heads, D=64, page 256, L=1536,
split 8) and the FlashMLA walk-through (656-byte FP8 token, section
"数据加载").
"""
from dataclasses import dataclass, field, replace
from typing import Optional, Sequence

# kv dtype tags (mirrors da_kv_dtype in include/decode_attn.h; plain ints so
# that this module holds no dependency on the library)
KV_BF16 = 0
KV_FP8 = 1
KV_MLA656 = 2


@dataclass(frozen=True)
class WorkloadSpec:
    name: str
    B: int
    H_kv: int
    G: int
    D_qk: int
    D_v: int
    page_size: int
    kv_dtype: int = KV_BF16
    # sequence lengths: either a fixed list, or a distribution recipe
    lengths: Optional[Sequence[int]] = None
    length_dist: str = "fixed"          # fixed | uniform | loguniform
    length_lo: int = 0
    length_hi: int = 0
    splits: int = 0                     # 0 = auto (balanced over SMs)
    extra_pages: int = 0                # unused pages in the pool (poisoned)
    softmax_scale: float = 0.0          # 0 = 1/sqrt(D_qk)
    seed: int = 0
    s_q: int = 1                        # query tokens per request (draft tokens of a linear chain)
    window: int = 0                     # sliding window in tokens (0: none)
    sinks: bool = False                 # one attention-sink logit per query head
    topk: int = 0                       # sparse decode: token positions listed per request (0: dense)
    description: str = field(default="", compare=False)

    @property
    def H_q(self) -> int:
        return self.H_kv * self.G

    def with_(self, **kw) -> "WorkloadSpec":
        return replace(self, **kw)


CONFIGS = [
    WorkloadSpec(
        name="tiny_gqa_bf16", B=1, H_kv=1, G=8, D_qk=64, D_v=64, page_size=16,
        lengths=[256], splits=1, extra_pages=48, seed=1000,
        description="B=1 H_q=8 H_kv=1 D=64 L=256 P=16, 64-page pool, splits=1"),
    WorkloadSpec(
        name="gqa_bf16_b8", B=8, H_kv=4, G=8, D_qk=64, D_v=64, page_size=256,
        lengths=[1536] * 8, splits=8, seed=1001,
        description="B=8 H_q=32 H_kv=4 D=64 P=256 L=1536 splits=8 (MetaX shape, batch 8)"),
    WorkloadSpec(
        name="mixed_gqa_bf16", B=32, H_kv=8, G=8, D_qk=128, D_v=128, page_size=64,
        length_dist="uniform", length_lo=1024, length_hi=8192, splits=0, seed=1002,
        description="B=32 H_q=64 H_kv=8 D=128 P=64 L~U[1024,8192] auto splits"),
    WorkloadSpec(
        name="fp8_gqa", B=64, H_kv=4, G=8, D_qk=128, D_v=128, page_size=32,
        kv_dtype=KV_FP8, lengths=[32768] * 64, splits=0, seed=1003,
        description="B=64 H_q=32 H_kv=4 D=128 P=32 L=32768 e4m3 KV, per-(head,tensor) fp32 scales"),
    WorkloadSpec(
        name="mla_fp8", B=32, H_kv=1, G=128, D_qk=576, D_v=512, page_size=64,
        kv_dtype=KV_MLA656, length_dist="loguniform", length_lo=4096, length_hi=131072,
        splits=0, seed=1004,
        description="B=32 H_q=128 H_kv=1 D_qk=576 D_v=512 P=64 656-byte FP8 tokens, "
                    "L log-uniform [4096,131072]"),
    # several query tokens per request (a chain of drafts being verified); not
    # a shape the pages measure: the mixed and FP8 shapes with s_q = 2 and 4
    WorkloadSpec(
        name="spec2_gqa_bf16", B=32, H_kv=8, G=8, D_qk=128, D_v=128, page_size=64,
        length_dist="uniform", length_lo=1024, length_hi=8192, splits=0, seed=1005, s_q=2,
        description="B=32 s_q=2 H_q=64 H_kv=8 D=128 P=64 L~U[1024,8192] auto splits, draft chain of 2"),
    WorkloadSpec(
        name="spec2_fp8_gqa", B=64, H_kv=4, G=8, D_qk=128, D_v=128, page_size=32,
        kv_dtype=KV_FP8, lengths=[32768] * 64, splits=0, seed=1006, s_q=2,
        description="B=64 s_q=2 H_q=32 H_kv=4 D=128 P=32 L=32768 e4m3 KV, draft chain of 2"),
    WorkloadSpec(
        name="spec4_gqa_d64", B=32, H_kv=8, G=8, D_qk=64, D_v=64, page_size=64,
        length_dist="uniform", length_lo=1024, length_hi=8192, splits=0, seed=1007, s_q=4,
        description="B=32 s_q=4 H_q=64 H_kv=8 D=64 P=64 L~U[1024,8192] auto splits, draft chain of 4"),
    WorkloadSpec(
        name="spec4_gqa_bf16", B=32, H_kv=8, G=8, D_qk=128, D_v=128, page_size=64,
        length_dist="uniform", length_lo=1024, length_hi=8192, splits=0, seed=1010, s_q=4,
        description="B=32 s_q=4 H_q=64 H_kv=8 D=128 P=64 L~U[1024,8192] auto splits, draft chain of 4"),
    # sliding window and attention sinks (the pages name both; no measured shape)
    WorkloadSpec(
        name="window_sinks_gqa_bf16", B=32, H_kv=8, G=8, D_qk=128, D_v=128, page_size=64,
        length_dist="uniform", length_lo=1024, length_hi=8192, splits=0, seed=1008, window=2048, sinks=True,
        description="B=32 H_q=64 H_kv=8 D=128 P=64 L~U[1024,8192] sliding window 2048, one sink per head"),
    # the latent-token workload with two query tokens per request (FlashMLA's call
    # passes s_q * h_q / h_kv rows per KV head; no page gives a number for it)
    WorkloadSpec(
        name="spec2_mla_fp8", B=32, H_kv=1, G=128, D_qk=576, D_v=512, page_size=64,
        kv_dtype=KV_MLA656, length_dist="loguniform", length_lo=4096, length_hi=131072,
        splits=0, seed=1011, s_q=2,
        description="B=32 s_q=2 H_q=128 H_kv=1 D_qk=576 D_v=512 P=64 656-byte FP8 tokens, "
                    "L log-uniform [4096,131072], draft chain of 2"),
    # sparse top-k decode on the latent-token format: the pages' "FP8 稀疏解码" row
    # (topk 2048, batch 128, 128 heads); the context length is not given there
    WorkloadSpec(
        name="sparse_mla_topk2048", B=128, H_kv=1, G=128, D_qk=576, D_v=512, page_size=64,
        kv_dtype=KV_MLA656, lengths=[8192] * 128, splits=0, seed=1009, topk=2048,
        description="B=128 H_q=128 656-byte FP8 tokens, L=8192, top-k 2048 positions per request"),
    # the same row's top-k 32768 figure; the page gives neither batch nor context,
    # so this takes the dense latent workload's batch and a context of twice top-k
    WorkloadSpec(
        name="sparse_mla_topk32768", B=32, H_kv=1, G=128, D_qk=576, D_v=512, page_size=64,
        kv_dtype=KV_MLA656, lengths=[65536] * 32, splits=0, seed=1012, topk=32768,
        description="B=32 H_q=128 656-byte FP8 tokens, L=65536, top-k 32768 positions per request"),
]


def spec_by_name(name: str) -> WorkloadSpec:
    for s in CONFIGS:
        if s.name == name:
            return s
    raise KeyError(name)
