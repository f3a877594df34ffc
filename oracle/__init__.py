"""CPU oracle (test infrastructure only): fp64 restatement of the unmerged multi-adapter LoRA layer."""
from .lora_oracle import (OK, EINVAL, ENOPAGES, EUNKNOWN_ADAPTER, ERANK, EEXIST, EBUSY, MAX_RANK,  # noqa: F401
                          EVICT_LOAD_ORDER, EVICT_LRU, EVICT_FARTHEST,
                          PoolModel, bf16_to_f64, bf16_round, gather_adapter, linear_forward, place_adapter,
                          merged_forward, segments, attention_decode)
