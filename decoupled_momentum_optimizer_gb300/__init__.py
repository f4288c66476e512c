"""GB300-native decoupled-momentum (DeMo / FlexDeMo) shard step."""
