"""KV-cache sizing closed forms -- TEST INFRASTRUCTURE ONLY (part of the oracle).

Each function writes out a sizing rule the pages state:

* KV bytes per token = 2 (K and V) * layers * hidden * dtype_bytes
  (studying-code.tistory.com/16, section "vLLM의 기존 문제점 - 비효율적인 KV캐시
  메모리 관리": about 800 KB per token for OPT-13B and about 1.6 GB for a
  2048-token request; OPT-13B has 40 layers and hidden size 5120).
* page size of one block = (K+V) * block_size * num_kv_heads * head_size * dtype_bytes
  (itan.pw "vLLMにおけるKVCacheマネージャーの詳細解説", section
  "ブロックアロケーションの基本概念"; 8192 bytes for the Qwen2-0.5B spec of section
  "BlockPoolの生成過程": block_size 16, 2 KV heads, head size 64, bf16).
* bytes of one layer's cache tensor = page_size * num_blocks
  (same page, section "BlockPoolの生成過程": 1080754176 = 8192 x 131928).
* blocks for n tokens = ceil(n / block_size)
  (same page, section "ブロック割当のロジック": cdiv(num_tokens, block_size),
  10 tokens at block size 16 take one block; and "ブロックアロケーションの基本概念":
  5 tokens take one block).
"""
from __future__ import annotations


def kv_bytes_per_token(num_layers: int, hidden_size: int, dtype_bytes: int) -> int:
    return 2 * num_layers * hidden_size * dtype_bytes


def page_size_bytes(block_size: int, num_kv_heads: int, head_size: int,
                    dtype_bytes: int) -> int:
    return 2 * block_size * num_kv_heads * head_size * dtype_bytes


def layer_tensor_bytes(page_size: int, num_blocks: int) -> int:
    return page_size * num_blocks


def cache_shape(num_blocks: int, block_size: int, num_kv_heads: int, head_size: int):
    return (2, num_blocks, block_size, num_kv_heads, head_size)


def blocks_for_tokens(num_tokens: int, block_size: int) -> int:
    return -(-num_tokens // block_size)
